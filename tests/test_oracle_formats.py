"""Pins for the oracle's alternate receive formats (CPU only).

Pre-encoded input (DeepEP "Normal Mode API", Quantization: x given as a
(data, scale) tuple of MXFP8 / MXFP4 rows): dispatch moves each source row's
bytes unchanged.  Pinned two ways: against brute force on random bytes, and
against the fused dispatch -- encoding every source row first and then moving
the bytes must give exactly the rows the fused dispatch writes.

Block-major scales (Modular MAX "EPBatchManager", ep_dispatch returns: FP8
output_scales of shape (hidden // block_size, max_recv_tokens)): element b of
receive row r sits at [b, r].  Pinned by hand-written examples and by the
identity that reading it back column by column gives the row-major scales.

Two-phase form (Modular MAX ep_dispatch_async / wait, ep_combine_async /
wait): the return slots against brute force, the wait phase over them equal
to the one-call combine, and the arrival rows of the per-rank layout expanded
by the grouped layout equal to the fused dispatch.
"""
import numpy as np
import pytest

import oracle
from combine_ep_layout_03_gb300 import synth


def brute_bytes(dst_row, src, rows):
    N, nb = src.shape
    K = dst_row.size // max(N, 1) if N else 1
    out = np.zeros((rows, nb), np.uint8)
    hit = np.zeros(rows, bool)
    for n in range(N):
        for k in range(K):
            d = int(dst_row.reshape(N, K)[n, k])
            if d >= 0:
                assert not hit[d]
                hit[d] = True
                out[d] = src[n]
    return out


@pytest.mark.parametrize("seed", range(12))
def test_dispatch_bytes_brute_force(seed):
    rng = np.random.default_rng(900 + seed)
    R, L = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    E = R * L
    K = int(rng.integers(1, min(E, 4) + 1))
    T = int(rng.integers(0, 7))
    alpha = int(rng.integers(1, 5))
    nb = int(rng.choice([1, 4, 7, 16, 33]))
    topk = rng.integers(-1, E, size=(R, T, K))
    src = rng.integers(0, 256, size=(R * T, nb), dtype=np.uint8)
    lay = oracle.layout(R, T, E, K, alpha, topk)
    got = oracle.dispatch_bytes(lay, src)
    assert np.array_equal(got, brute_bytes(lay.dst_row, src, lay.rows))
    # padding rows (recv_src = -1) are zero
    assert not got[lay.recv_src < 0].any()
    # the per-rank layout moves the same bytes onto its own rows
    w = rng.random((R, T, K)).astype(np.float32)
    tl = oracle.token_layout(R, T, E, K, topk, w)
    got_t = oracle.dispatch_bytes(tl, src)
    assert np.array_equal(got_t, src[tl.recv_src])


@pytest.mark.parametrize("q", [oracle.Q_NONE, oracle.Q_INT8, oracle.Q_E4M3, oracle.Q_E5M2,
                               oracle.Q_E2M1, oracle.Q_FP8T_E4M3, oracle.Q_FP8G_E5M2])
def test_encode_then_move_equals_fused_dispatch(q):
    w = synth.WORKLOADS[1].with_(H=256, alpha=4)
    topk = synth.gen_topk(w)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    N = w.R * w.T
    db, sb = oracle.row_bytes(q, w.H)
    src_d = np.zeros((N, db), np.uint8)
    src_s = np.zeros((N, sb), np.uint8)
    xr = x.reshape(N, w.H)
    for n in range(N):
        src_d[n], src_s[n] = oracle.encode_row(q, xr[n])
    fused_d, fused_s = oracle.dispatch(lay, x, q)
    assert np.array_equal(oracle.dispatch_bytes(lay, src_d), fused_d)
    if sb:
        assert np.array_equal(oracle.dispatch_bytes(lay, src_s), fused_s)


@pytest.mark.parametrize("q", [oracle.Q_NONE, oracle.Q_INT8, oracle.Q_E4M3, oracle.Q_E2M1,
                               oracle.Q_FP8G_E4M3])
@pytest.mark.parametrize("threads", [1, 3])
def test_encode_rows_then_ranked_moves_equal_fused_dispatch(q, threads):
    """The batch encoder with a rank-by-rank scatter (as the full-size GPU
    parity builds the receive buffer) equals the oracle's fused dispatch."""
    w = synth.WORKLOADS[3].with_(T=40, H=256)       # Zipf routing, alpha = 128: padding rows
    topk = synth.gen_topk(w)
    x = synth.gen_x(w).reshape(w.R * w.T, w.H)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    enc_d, enc_s = oracle.encode_rows(q, x, threads)
    for n in (0, 7, w.R * w.T - 1):
        d1, s1 = oracle.encode_row(q, x[n])
        assert np.array_equal(enc_d[n], d1) and np.array_equal(enc_s[n], s1)
    fused_d, fused_s = oracle.dispatch(lay, x, q)
    db, sb = oracle.row_bytes(q, w.H)
    for j in range(w.R):
        a, b = int(lay.rank_base[j]), int(lay.rank_base[j + 1])
        buf = np.full((b - a, db), 0xA5, np.uint8)
        oracle.dispatch_bytes(lay, enc_d, rows=b, row_begin=a, out=buf)
        assert np.array_equal(buf, fused_d[a:b])
        if sb:
            assert np.array_equal(oracle.dispatch_bytes(lay, enc_s, rows=b, row_begin=a), fused_s[a:b])


def test_transpose_scales_hand_worked():
    rows = np.array([[1, 2, 3], [4, 5, 6]], np.uint8)
    expect = np.array([[1, 4, 0, 0], [2, 5, 0, 0], [3, 6, 0, 0]], np.uint8)
    assert np.array_equal(oracle.transpose_scales(rows, 4, 1), expect)
    # float32 elements: whole 4-byte words move together
    f = np.array([[1.5, -2.0], [0.25, 8.0], [3.0, 0.5]], np.float32)
    got = oracle.transpose_scales(f.view(np.uint8).reshape(3, 8), 5, 4).view(np.float32)
    assert np.array_equal(got, np.array([[1.5, 0.25, 3.0, 0, 0], [-2.0, 8.0, 0.5, 0, 0]], np.float32))
    # one scale per row (per-token modes): the same bytes, padded to the capacity
    t = np.array([[9, 8, 7, 6], [5, 4, 3, 2]], np.uint8)
    assert np.array_equal(oracle.transpose_scales(t, 3, 4), np.array([[9, 8, 7, 6, 5, 4, 3, 2, 0, 0, 0, 0]], np.uint8))


@pytest.mark.parametrize("elem", [1, 4])
def test_transpose_scales_reads_back(elem):
    rng = np.random.default_rng(elem)
    rows, nb, cap = 37, 6, 50
    s = rng.integers(0, 256, size=(rows, nb * elem), dtype=np.uint8)
    t = oracle.transpose_scales(s, cap, elem).reshape(nb, cap, elem)
    for r in range(rows):
        for b in range(nb):
            assert np.array_equal(t[b, r], s[r, b * elem:(b + 1) * elem])
    assert not t[:, rows:].any()


# ---- two-phase form (MAX ep_dispatch_async / wait, ep_combine_async / wait) ----

def test_return_slots_brute_force_and_wait_equals_combine():
    rng = np.random.default_rng(31)
    R, T, E, K, H = 3, 5, 6, 3, 16
    topk = rng.integers(-1, E, size=(R, T, K))
    lay = oracle.layout(R, T, E, K, 2, topk)
    y = rng.integers(0, 1 << 15, size=(max(lay.rows, 1), H), dtype=np.uint16)   # finite bf16 patterns
    slots, valid = oracle.return_slots(lay, y)
    for s in range(R):
        for t in range(T):
            for k in range(K):
                i = (s * T + t) * K + k
                d = int(lay.dst_row[s, t, k])
                assert valid[i] == (d >= 0)
                if d >= 0:
                    assert np.array_equal(slots[i], y[d])
    w = rng.random((R, T, K)).astype(np.float32)
    # the wait phase over the slots reproduces the one-call combine exactly
    assert np.array_equal(oracle.combine(oracle.slot_layout(lay), slots, w), oracle.combine(lay, y, w))


def test_dispatch_wait_of_arrival_rows_equals_dispatch():
    # arrival rows (per-rank layout) expanded by the grouped layout's rows are the fused dispatch
    w = synth.WORKLOADS[1].with_(H=128, alpha=4, T=20)
    topk = synth.gen_topk(w)
    wts = synth.gen_weights(w, topk)
    x = synth.gen_x(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    tl = oracle.token_layout(w.R, w.T, w.E, w.K, topk, wts)
    for q in (oracle.Q_NONE, oracle.Q_E4M3, oracle.Q_INT8):
        td, ts = oracle.token_dispatch(tl, x, q)
        # per grouped row: the arrival row of its source token on its rank
        rank_of_row = np.searchsorted(lay.rank_base, np.arange(lay.rows), side="right") - 1
        src = lay.recv_src
        d, s_ = oracle.dispatch(lay, x, q)
        for r in range(lay.rows):
            if src[r] < 0:
                assert not d[r].any()
                continue
            j = rank_of_row[r]
            p = [q_ for q_ in tl.tok_dst[src[r]] if tl.rank_tok_base[j] <= q_ < tl.rank_tok_base[j + 1]]
            assert len(p) == 1
            assert np.array_equal(td[p[0]], d[r])
            if s_.shape[1]:
                assert np.array_equal(ts[p[0]], s_[r])
