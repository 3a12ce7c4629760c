"""The allocation-free layout entry point (ep_layout_static_scratch).

It serves callers that can pass output buffers but cannot allocate device
memory themselves while they run.  The test calls it through the C ABI with
outputs the test allocates, several times in a row on problems of different
sizes (so a later call runs over the previous call's leftovers in the shared
static scratch array), and checks every output against the ordinary ep_layout
entry point bit for bit (layout results are integers: the parity bar is
exact equality).  This file is collected last.
"""
import numpy as np
import pytest
import torch

from combine_ep_layout_03_gb300 import ep, synth

pytestmark = pytest.mark.gpu

SHAPES = {
    "status": (torch.int32, lambda w: (1,)),
    "cnt": (torch.int32, lambda w: (w.R, w.E)),
    "is_token_in_rank": (torch.uint8, lambda w: (w.R, w.T, w.R)),
    "num_tokens_per_rank": (torch.int32, lambda w: (w.R, w.R)),
    "recv_cnt": (torch.int32, lambda w: (w.E,)),
    "aligned_cnt": (torch.int32, lambda w: (w.R, w.L)),
    "expert_start": (torch.int32, lambda w: (w.R, w.L + 1)),
    "rank_base": (torch.int64, lambda w: (w.R + 1,)),
    "expert_base": (torch.int32, lambda w: (w.E + 1,)),
    "src_prefix": (torch.int32, lambda w: (w.R, w.E)),
    "dst_row": (torch.int32, lambda w: (w.R, w.T, w.K)),
    "recv_src": (torch.int32, lambda w: (w.N * w.K + w.E * (w.alpha - 1),)),
    "expert_ids": (torch.int32, lambda w: (w.R, w.L)),
    "expert_usage_stats": (torch.int32, lambda w: (w.R, 2)),
}


def outputs_for(w):
    outs = {}
    for name, (dt, shape) in SHAPES.items():
        t = torch.empty(shape(w), dtype=dt, device="cuda")
        t.fill_(0x5A if dt == torch.uint8 else -7)   # garbage the call must overwrite
        outs[name] = t
    return outs


def reference_layout(w, topk_dev):
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha)
    lay.layout(topk_dev)
    views = {k: v.clone() for k, v in lay.views().items()}
    status = lay.status()
    rows = lay.recv_rows()[-1]
    return views, status, rows


def check_against_reference(w, topk):
    topk_dev = torch.from_numpy(np.ascontiguousarray(topk)).cuda()
    params = ep.make_params(w.R, w.T, w.H, w.E, w.K, w.alpha, 0)
    outs = outputs_for(w)
    ep.ep_layout_static_scratch(params, topk_dev, outs)
    torch.cuda.synchronize()
    ref, ref_status, rows = reference_layout(w, topk_dev)
    assert int(outs["status"].item()) == ref_status
    for name in SHAPES:
        if name in ("status", "recv_src"):
            continue
        assert torch.equal(outs[name], ref[name]), name
    assert torch.equal(outs["recv_src"][:rows], ref["recv_src"][:rows])
    return ref_status


def test_static_scratch_layout_matches_ep_layout_on_calls_in_a_row():
    small = synth.WORKLOADS[1]
    wide = synth.WORKLOADS[5].with_(T=200)       # 32 ranks, 512 experts, K=16, 10% -1
    skew = synth.WORKLOADS[3].with_(T=300)       # Zipf routing, alpha = 128
    assert check_against_reference(small, synth.gen_topk(small)) == ep.EP_OK
    assert check_against_reference(wide, synth.gen_topk(wide)) == ep.EP_OK
    assert check_against_reference(skew, synth.gen_topk(skew)) == ep.EP_OK
    assert check_against_reference(small, synth.gen_topk(small)) == ep.EP_OK


def test_static_scratch_reports_bad_ids_and_oversize():
    w = synth.WORKLOADS[1]
    topk = synth.gen_topk(w)
    topk[1, 3, 0] = 99
    assert check_against_reference(w, topk) == ep.EP_ERR_BAD_EXPERT_ID
    # scratch beyond the 2 MiB maximum is refused on the host
    big = synth.Workload(20, R=512, T=64, H=64, E=512, K=2, alpha=1)
    outs = outputs_for(big)
    topk_dev = torch.zeros((big.R, big.T, big.K), dtype=torch.int64, device="cuda")
    with pytest.raises(ep.EPError) as ei:
        ep.ep_layout_static_scratch(ep.make_params(big.R, big.T, big.H, big.E, big.K, 1, 0),
                                    topk_dev, outs)
    assert ei.value.status == ep.EP_ERR_UNSUPPORTED
