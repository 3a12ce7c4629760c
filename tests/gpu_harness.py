"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
on seeded inputs, and compare with the CPU oracle."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from combine_ep_layout_03_gb300 import synth

LAYOUT_KEYS = ("cnt", "is_token_in_rank", "num_tokens_per_rank", "recv_cnt", "expert_start",
               "rank_base", "src_prefix", "dst_row", "expert_usage_stats", "expert_ids")


def to_dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(dev).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GpuPath:
    """Layout + dispatch (+ stand-in expert + combine) on the GPU."""

    def __init__(self, w: synth.Workload, topk: np.ndarray, recv_capacity_rows: int = 0):
        from combine_ep_layout_03_gb300 import ep
        self.ep = ep
        self.w = w
        self.lay = ep.EPLayout(w.R, w.T, w.H, w.E, w.K, w.alpha, recv_capacity_rows)
        self.topk_dev = torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int64)).cuda()
        self.lay.layout(self.topk_dev)
        self.rank_base = self.lay.recv_rows()
        self.rows = int(self.rank_base[-1])

    def views_numpy(self) -> dict:
        v = self.lay.views()
        out = {k: t.cpu().numpy() for k, t in v.items()}
        out["recv_src"] = out["recv_src"][: min(self.rows, self.lay.recv_src_capacity)]
        return out

    def dispatch(self, x_dev: torch.Tensor, quant: int, rows: int | None = None,
                 fill: int | None = None):
        rows = max(self.rows, 1) if rows is None else rows
        data, scales = self.lay.alloc_recv(quant, rows)
        if fill is not None:
            data.fill_(fill)
            if scales is not None:
                scales.fill_(fill)
        self.lay.dispatch(x_dev, quant, data, scales)
        return data, scales

    def expert(self, quant: int, data, scales, mark_mod: int, inplace: bool = False):
        rows = data.shape[0]
        if inplace and quant == 0:
            y = data.view(torch.bfloat16).view(rows, self.w.H)
        else:
            y = torch.empty((rows, self.w.H), dtype=torch.bfloat16, device="cuda")
        self.lay.expert_identity(quant, data, scales, y, mark_mod)
        return y

    def combine(self, y, wts_dev, shared_dev=None):
        out = torch.empty((self.w.N, self.w.H), dtype=torch.bfloat16, device="cuda")
        self.lay.combine(y, wts_dev, out, shared_dev)
        return out


def compare_layout(g: dict, olay: oracle.Layout):
    for k in LAYOUT_KEYS:
        a, b = g[k], getattr(olay, k)
        assert a.shape == b.shape or a.size == b.size, (k, a.shape, b.shape)
        assert np.array_equal(a.reshape(b.shape), b), f"layout mismatch in {k}"
    assert np.array_equal(g["aligned_cnt"].reshape(-1), olay.aligned)
    assert np.array_equal(g["recv_cnt"], olay.recv_cnt)
    eb = np.concatenate([[0], np.cumsum(olay.aligned)])
    assert np.array_equal(g["expert_base"], eb)
    assert np.array_equal(g["recv_src"], olay.recv_src), "layout mismatch in recv_src"


def y_rows_for_tokens(olay: oracle.Layout, tokens: np.ndarray):
    """Receive rows used by a set of source tokens, and a map row -> index."""
    d = olay.dst_row.reshape(-1, olay.K)[tokens].reshape(-1)
    rows = np.unique(d[d >= 0])
    ymap = np.full(max(olay.rows, 1), -1, np.int64)
    ymap[rows] = np.arange(len(rows))
    return rows, ymap


def oracle_combine_sampled(olay, x_bits, wts, shared_tok, quant, mark_mod, tokens):
    """Oracle combine of selected source tokens, with the oracle's own dispatch
    and stand-in expert.  shared_tok: [len(tokens), S, H] bf16 bits or None (the
    shared-expert rows of just those tokens).  Each token is combined through a
    one-token layout (R = T = 1) that keeps its dst_row entries, so only the
    sampled shared rows need to be on the host."""
    K = olay.K
    H = x_bits.shape[-1]
    rows, ymap = y_rows_for_tokens(olay, tokens)
    data, scales = oracle.dispatch_rows(olay, x_bits, quant, rows)
    y = oracle.expert_rows(olay, rows, H, quant, data, scales, mark_mod)
    dr = olay.dst_row.reshape(-1, K)
    wf = np.asarray(wts, np.float32).reshape(-1, K)
    outs, refs, mags = [], [], []
    for i, n in enumerate(tokens):
        mini = oracle.Layout(R=1, T=1, K=K, dst_row=np.ascontiguousarray(dr[n].reshape(1, 1, K)))
        sh = None if shared_tok is None else np.ascontiguousarray(shared_tok[i][None, :, None, :])
        outs.append(oracle.combine(mini, y, wf[n], sh, 0, 1, ymap))
        r, m = oracle.combine_ref64(mini, y, wf[n], sh, 0, 1, ymap)
        refs.append(r)
        mags.append(m)
    return np.concatenate(outs), np.concatenate(refs), np.concatenate(mags)


def host_threads(cap: int = 16) -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    return max(1, min(cap, n))


def for_row_chunks(total: int, fn, step: int = 32768, threads: int | None = None):
    """Run fn(a, b) over [0, total) in chunks of `step` rows on host threads
    (the oracle's C calls release the interpreter lock); re-raises the first
    failure."""
    if total <= 0:
        return
    with ThreadPoolExecutor(max_workers=threads or host_threads()) as ex:
        list(ex.map(lambda a: fn(a, min(total, a + step)), range(0, total, step)))
