"""The allocation-free layout entry point (ep_layout_static_scratch).

It serves callers that can pass output buffers but cannot allocate device
memory themselves while they run.  The test calls it through the C ABI with
outputs the test allocates, several times in a row on problems of different
sizes (so a later call runs over the previous call's leftovers in the shared
static scratch array), and checks every output bit for bit both against the
ordinary ep_layout entry point and against the CPU oracle's layout (layout
results are integers: the parity bar is exact equality).  It also covers a
receive capacity that the routing overflows (status EP_ERR_CAPACITY, recv_src
written only below the capacity) and a call on a stream other than the
default one.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
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


GUARD = 64   # recv_src entries past the capacity that no call may write


def outputs_for(w, cap=0):
    outs = {}
    for name, (dt, shape) in SHAPES.items():
        shp = (cap + GUARD,) if (name == "recv_src" and cap) else shape(w)
        t = torch.empty(shp, dtype=dt, device="cuda")
        t.fill_(0x5A if dt == torch.uint8 else -7)   # garbage the call must overwrite
        outs[name] = t
    return outs


def reference_layout(w, topk_dev, cap=0):
    lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha, cap)
    lay.layout(topk_dev)
    views = {k: v.clone() for k, v in lay.views().items()}
    status = lay.status()
    rows = lay.recv_rows()[-1]
    return views, status, rows


def check_against_oracle(w, topk, outs, cap=0):
    olay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk, recv_cap=cap or None)
    got = {k: v.cpu().numpy() for k, v in outs.items()}
    assert int(got["status"][0]) == olay.status
    for name in ("cnt", "is_token_in_rank", "num_tokens_per_rank", "recv_cnt", "expert_start",
                 "rank_base", "src_prefix", "dst_row", "expert_ids", "expert_usage_stats"):
        assert np.array_equal(got[name].reshape(getattr(olay, name).shape), getattr(olay, name)), name
    assert np.array_equal(got["aligned_cnt"].reshape(-1), olay.aligned)
    assert np.array_equal(got["expert_base"], np.concatenate([[0], np.cumsum(olay.aligned)]))
    n = len(olay.recv_src)   # rows below the capacity
    assert np.array_equal(got["recv_src"][:n], olay.recv_src)
    return olay


def check_against_reference(w, topk, cap=0, stream=None):
    topk_dev = torch.from_numpy(np.ascontiguousarray(topk)).cuda()
    params = ep.make_params(w.R, w.T, w.H, w.E, w.K, w.alpha, cap)
    outs = outputs_for(w, cap)
    torch.cuda.synchronize()
    if stream is None:
        ep.ep_layout_static_scratch(params, topk_dev, outs)
    else:
        with torch.cuda.stream(stream):
            ep.ep_layout_static_scratch(params, topk_dev, outs, stream)
    torch.cuda.synchronize()
    ref, ref_status, rows = reference_layout(w, topk_dev, cap)
    assert int(outs["status"].item()) == ref_status
    for name in SHAPES:
        if name in ("status", "recv_src"):
            continue
        assert torch.equal(outs[name], ref[name]), name
    n = min(rows, cap) if cap else rows
    assert torch.equal(outs["recv_src"][:n], ref["recv_src"][:n])
    if cap:
        # nothing is written past the capacity
        assert torch.all(outs["recv_src"][cap:] == -7)
    check_against_oracle(w, topk, outs, cap)
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


def test_static_scratch_capacity_overflow_writes_nothing_past_the_capacity():
    w = synth.WORKLOADS[3].with_(T=64)            # Zipf routing, alpha = 128: many padding rows
    topk = synth.gen_topk(w)
    rows = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk).rows
    cap = rows // 2
    assert check_against_reference(w, topk, cap=cap) == ep.EP_ERR_CAPACITY
    # a capacity that fits exactly is not an overflow
    assert check_against_reference(w, topk, cap=rows) == ep.EP_OK


def test_static_scratch_on_a_side_stream():
    w = synth.WORKLOADS[2].with_(T=96)
    topk = synth.gen_topk(w)
    side = torch.cuda.Stream()
    assert check_against_reference(w, topk, stream=side) == ep.EP_OK
    assert check_against_reference(w, topk) == ep.EP_OK
