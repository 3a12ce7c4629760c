"""GPU parity for the DeepEP per-rank receive layout (one row per token and
destination rank; recv_topk_idx / recv_topk_weights; combine of per-rank rows
with reduced weights) against the oracle.

Bit-exact: tok_dst, recv_src_tok, rank_tok_base, recv_topk_idx,
recv_topk_weights, receive rows and scales, the per-rank stand-in expert
stage, and the reduced weights (both sum in ascending rank order).  Combine:
within the derived tolerance.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_03_gb300 import ep, synth
from gpu_harness import bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


def run_tokens(w, q=0, mark=4, mask_dims=0, check_all_rows=True):
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    mask = synth.gen_mask(w, mask_dims) if mask_dims else None
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts, mask=mask)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    w_d = torch.from_numpy(wts).cuda()
    mask_d = None if mask is None else torch.from_numpy(mask).cuda()
    lay.layout(topk_d, active_mask=mask_d)
    ridx, rw = lay.token_layout(topk_d, w_d, active_mask=mask_d)
    base = lay.token_rows()
    assert base[-1] == tl.rows and lay.status() == 0
    v = lay.views()
    assert np.array_equal(v["tok_dst"].cpu().numpy().reshape(w.N, w.K), tl.tok_dst)
    assert np.array_equal(v["rank_tok_base"].cpu().numpy(), tl.rank_tok_base)
    assert np.array_equal(v["recv_src_tok"][: tl.rows].cpu().numpy(), tl.recv_src)
    assert np.array_equal(ridx[: tl.rows].cpu().numpy(), tl.recv_topk_idx)
    assert np.array_equal(rw[: tl.rows].cpu().numpy(), tl.recv_topk_weights)
    # dispatch into the per-rank layout
    data, sc = lay.alloc_recv(q, max(tl.rows, 1))
    data.fill_(0x3C)
    lay.dispatch_tokens(to_dev_bf16(x), q, data, sc)
    od, os_ = oracle.token_dispatch(tl, x, q)
    assert np.array_equal(data[: tl.rows].cpu().numpy(), od)
    if os_.shape[1]:
        assert np.array_equal(sc[: tl.rows].cpu().numpy(), os_)
    # stand-in expert stage of each rank, then combine with reduced weights
    y = torch.empty((max(tl.rows, 1), w.H), dtype=torch.bfloat16, device="cuda")
    lay.expert_identity_tokens(q, data, sc, ridx, rw, y, mark)
    oy = oracle.expert_token_rows(tl, w.H, q, od, os_, mark)
    assert np.array_equal(bf16_bits(y[: tl.rows]), oy), "per-rank expert stage differs"
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    out_w = torch.empty((w.N, w.K), dtype=torch.float32, device="cuda")
    sh_d = None if shared is None else to_dev_bf16(shared)
    lay.combine_tokens(y, out, sh_d, rank_weights=rw, out_weights=out_w)
    ref, mag = oracle.token_combine_ref64(tl, oy, shared)
    ok, excess, rel = oracle.combine_within_tolerance(bf16_bits(out), ref, mag, w.K, w.num_shared)
    assert ok, (excess, rel)
    assert np.array_equal(out_w.cpu().numpy(), oracle.reduce_token_weights(tl, tl.recv_topk_weights))
    assert lay.status() == 0


@pytest.mark.parametrize("idx,T,q", [(1, 64, 0), (2, 300, 0), (5, 90, 0), (3, 100, 2), (4, 150, 4),
                                     (4, 150, 6), (4, 150, 9)])
def test_token_layout_dispatch_combine(idx, T, q):
    run_tokens(synth.WORKLOADS[idx].with_(T=T), q)


@pytest.mark.parametrize("dims", [1, 2])
def test_token_layout_with_mask(dims):
    run_tokens(synth.WORKLOADS[5].with_(T=60), 0, 8, dims)


def test_token_layout_edges():
    # T = 0, a single rank, K = 1, tokens without experts
    run_tokens(synth.Workload(30, R=3, T=0, H=64, E=6, K=2, alpha=1))
    run_tokens(synth.Workload(31, R=1, T=50, H=64, E=4, K=3, alpha=1))
    run_tokens(synth.Workload(32, R=4, T=40, H=128, E=8, K=1, alpha=1))
    run_tokens(synth.Workload(33, R=4, T=40, H=128, E=16, K=4, alpha=1, drop_p=0.6))


@pytest.mark.parametrize("idx,q", [(2, 0), (4, 4)])
def test_token_layout_full_size_every_row(idx, q):
    """Workloads 2 (bf16) and 4 (MXFP8 e4m3) at full size in the per-rank layout
    (the bench's keys 2r and 4r): the layout arrays, recv_topk_idx /
    recv_topk_weights and the reduced weights for every token, and every
    receive row and scale row, in chunks of rows on host threads, against the
    oracle's per-token encoding placed by its own tok_dst."""
    from concurrent.futures import ThreadPoolExecutor
    w = synth.WORKLOADS[idx]
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    topk_d = torch.from_numpy(topk).cuda()
    lay.layout(topk_d)
    ridx, rw = lay.token_layout(topk_d, torch.from_numpy(wts).cuda())
    assert lay.token_rows()[-1] == tl.rows
    v = lay.views()
    assert np.array_equal(v["tok_dst"].cpu().numpy().reshape(w.N, w.K), tl.tok_dst)
    assert np.array_equal(v["rank_tok_base"].cpu().numpy(), tl.rank_tok_base)
    assert np.array_equal(v["recv_src_tok"][: tl.rows].cpu().numpy(), tl.recv_src)
    assert np.array_equal(ridx[: tl.rows].cpu().numpy(), tl.recv_topk_idx)
    assert np.array_equal(rw[: tl.rows].cpu().numpy(), tl.recv_topk_weights)
    x_dev = synth.gen_x_device(w)
    x = bf16_bits(x_dev).reshape(w.N, w.H)
    data, sc = lay.alloc_recv(q, tl.rows)
    data.fill_(0x3C)
    if sc is not None:
        sc.fill_(0x3C)
    lay.dispatch_tokens(x_dev, q, data, sc)
    torch.cuda.synchronize()
    assert lay.status() == 0
    threads = max(1, min(16, len(os.sched_getaffinity(0))))
    enc_d, enc_s = oracle.encode_rows(q, x, threads)
    step = 32768

    def chunk(a):
        b = min(tl.rows, a + step)
        od = oracle.dispatch_bytes(tl, enc_d, rows=b, row_begin=a)
        assert np.array_equal(data[a:b].cpu().numpy(), od), f"receive rows {a}:{b} differ"
        if sc is not None:
            os_ = oracle.dispatch_bytes(tl, enc_s, rows=b, row_begin=a)
            assert np.array_equal(sc[a:b].cpu().numpy(), os_), f"receive scales {a}:{b} differ"

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(chunk, range(0, tl.rows, step)))
    # the per-rank expert stage and the combine with the reduced weights of every token
    y = torch.empty((tl.rows, w.H), dtype=torch.bfloat16, device="cuda")
    lay.expert_identity_tokens(q, data, sc, ridx, rw, y, 4)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device="cuda")
    out_w = torch.empty((w.N, w.K), dtype=torch.float32, device="cuda")
    lay.combine_tokens(y, out, None, rank_weights=rw, out_weights=out_w)
    torch.cuda.synchronize()
    assert lay.status() == 0
    assert np.array_equal(out_w.cpu().numpy(), oracle.reduce_token_weights(tl, tl.recv_topk_weights))
