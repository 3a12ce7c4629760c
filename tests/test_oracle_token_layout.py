"""Pins for the oracle's per-rank receive layout (DeepEP "Normal Mode API":
recv_x one row per received token, recv_topk_idx / recv_topk_weights as seen
by the receiving rank; combine sums a token's per-rank rows and returns the
reduced weights).  CPU only.

Brute force: per destination rank, the sorted list of source tokens with an
expert there.  Closed form: with each rank's expert stage applying its local
experts (identity, or marked by local expert id) weighted by the received
weights, the combined output equals x * sum_k w_k * mark_k.
"""
import numpy as np
import pytest

import oracle
from combine_ep_layout_03_gb300 import synth


def brute_tokens(R, T, E, K, topk, w):
    L = E // R
    tk = topk.reshape(R * T, K)
    wf = w.reshape(R * T, K)
    rows, src, idx, wts = [], [], [], []
    tok_dst = -np.ones((R * T, K), np.int64)
    fill = np.zeros(R * T, np.int64)
    base = [0]
    for j in range(R):
        for n in range(R * T):
            ks = [k for k in range(K) if 0 <= tk[n, k] < E and tk[n, k] // L == j]
            if not ks:
                continue
            r = len(src)
            tok_dst[n, fill[n]] = r
            fill[n] += 1
            src.append(n)
            idx.append([tk[n, k] - j * L if k in ks else -1 for k in range(K)])
            wts.append([wf[n, k] if k in ks else 0.0 for k in range(K)])
        base.append(len(src))
    return dict(rows=len(src), tok_dst=tok_dst, recv_src=np.array(src, np.int64),
                rank_tok_base=np.array(base), recv_topk_idx=np.array(idx, np.int64).reshape(-1, K),
                recv_topk_weights=np.array(wts, np.float32).reshape(-1, K))


def check(tl, ref):
    assert tl.rows == ref["rows"]
    for k in ("tok_dst", "recv_src", "rank_tok_base", "recv_topk_idx", "recv_topk_weights"):
        assert np.array_equal(np.asarray(getattr(tl, k)).reshape(np.shape(ref[k])), ref[k]), k


@pytest.mark.parametrize("seed", range(20))
def test_random_small_against_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    R, L = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    E = R * L
    K = int(rng.integers(1, min(E, 4) + 1))
    T = int(rng.integers(0, 7))
    topk = rng.integers(-1, E, size=(R, T, K))
    w = rng.random((R, T, K)).astype(np.float32)
    check(oracle.token_layout(R, T, E, K, topk, w), brute_tokens(R, T, E, K, topk, w))


@pytest.mark.parametrize("idx,T", [(1, 64), (2, 40), (5, 12)])
def test_workloads_against_brute_force_and_expert_layout(idx, T):
    w = synth.WORKLOADS[idx].with_(T=T)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    check(tl, brute_tokens(w.R, w.T, w.E, w.K, topk, wts))
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    # rows of rank j = tokens routed to j = column sums of num_tokens_per_rank
    assert np.array_equal(np.diff(tl.rank_tok_base), lay.num_tokens_per_rank.sum(axis=0))
    assert tl.rows == int(lay.is_token_in_rank.sum())


def test_mask_equals_minus_one_substitution():
    w = synth.WORKLOADS[5].with_(T=10)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    mask = synth.gen_mask(w, 2, 0.7)
    sub = topk.copy()
    sub[mask == 0] = -1
    a = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts, mask=mask)
    check(a, brute_tokens(w.R, w.T, w.E, w.K, sub, wts))


@pytest.mark.parametrize("q", [oracle.Q_NONE, oracle.Q_INT8, oracle.Q_E4M3, oracle.Q_FP8G_E4M3])
def test_token_rows_hold_the_encoded_source_row(q):
    w = synth.WORKLOADS[4].with_(T=12)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    data, scales = oracle.token_dispatch(tl, x, q)
    for r in range(tl.rows):
        d, s_ = oracle.encode_row(q, x.reshape(w.N, w.H)[tl.recv_src[r]]) if q >= 7 else (None, None)
        if d is None:
            lay = oracle.layout(w.R, w.T, w.E, w.K, 1, topk)
            d, s_ = oracle.dispatch_rows(lay, x, q, lay.dst_row.reshape(w.N, w.K)[tl.recv_src[r]][:1])
            d, s_ = d[0], s_[0]
        assert np.array_equal(data[r], d) and np.array_equal(scales[r], s_)


@pytest.mark.parametrize("idx,T,mark", [(1, 64, 0), (2, 24, 4), (5, 10, 8), (4, 16, 2)])
def test_combine_through_rank_expert_stage_closed_form(idx, T, mark):
    # bf16 rows; each rank's stage sums its local experts (identity, marked by local id)
    w = synth.WORKLOADS[idx].with_(T=T)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    shared = synth.gen_shared(w)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    data, scales = oracle.token_dispatch(tl, x, oracle.Q_NONE)
    y = oracle.expert_token_rows(tl, w.H, oracle.Q_NONE, data, scales, mark)
    out = oracle.bf16_bits_to_f64(oracle.token_combine(tl, y, shared))
    tk = topk.reshape(w.N, w.K)
    valid = tk >= 0
    m = np.where(valid, 2.0 ** -((np.where(valid, tk, 0) % w.L) % mark) if mark else 1.0, 0.0)
    xf = oracle.bf16_bits_to_f64(x.reshape(w.N, w.H))
    c = wts.reshape(w.N, w.K).astype(np.float64) * m * valid
    ref = xf * c.sum(1)[:, None]
    routed = np.abs(xf) * np.abs(c).sum(1)[:, None]
    mag = routed.copy()
    if shared is not None:
        sh = oracle.bf16_bits_to_f64(shared).transpose(0, 2, 1, 3).reshape(w.N, w.num_shared, w.H)
        ref = ref + sh.sum(1)
        mag = mag + np.abs(sh).sum(1)
    # two bf16 roundings: each rank's stage output (<= 2^-8 relative to its sum, whose
    # magnitudes add up to at most `routed`) and the combine (2 ulp + fp32 floor)
    bound = (2 * oracle.ulp_bf16(ref) + np.ldexp(routed, -8)
             + oracle.combine_tolerance_floor(mag, w.K, w.num_shared))
    assert np.all(np.abs(out - ref) <= bound)


def test_reduced_weights_equal_original_for_valid_entries():
    w = synth.WORKLOADS[5].with_(T=16)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    red = oracle.reduce_token_weights(tl, tl.recv_topk_weights)
    want = np.where(topk.reshape(w.N, w.K) >= 0, wts.reshape(w.N, w.K), 0.0)
    assert np.array_equal(red, want.astype(np.float32))
