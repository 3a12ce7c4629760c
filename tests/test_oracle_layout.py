"""Pins for the oracle's routing layout (CPU only).

The oracle computes the layout with running counters and prefix sums over
(source rank, token, slot).  The brute force here builds the same receive
layout a different way: it sorts every valid (expert, source rank, token,
slot) entry and walks the experts in order, padding each segment up to the
alignment.  Both follow the DeepEP "Normal Mode API" dispatch parameters
(num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert, topk_idx with
-1 = no expert, expert_alignment) and the CANN rule localExpertNum =
moeExpertNum / epWorldSize; the receive order (destination rank, local
expert, source rank, token) is the deterministic order the design fixes.
"""
import itertools

import numpy as np
import pytest

import oracle
from combine_ep_layout_03_gb300 import synth


def brute_layout(R, T, E, K, alpha, topk):
    topk = np.asarray(topk).reshape(R, T, K)
    L = E // R
    entries = sorted((int(topk[s, t, k]), s, t, k)
                     for s in range(R) for t in range(T) for k in range(K) if topk[s, t, k] >= 0)
    dst = -np.ones((R, T, K), np.int64)
    recv_src = []
    seg = {}
    row = 0
    for e in range(E):
        start = row
        for (ee, s, t, k) in entries:
            if ee == e:
                dst[s, t, k] = row
                recv_src.append(s * T + t)
                row += 1
        while (row - start) % alpha:
            recv_src.append(-1)
            row += 1
        seg[e] = (start, row)
    cnt = np.zeros((R, E), np.int64)
    for (e, s, t, k) in entries:
        cnt[s, e] += 1
    itr = np.zeros((R, T, R), np.int64)
    for s in range(R):
        for t in range(T):
            for j in {int(e) // L for e in topk[s, t] if e >= 0}:
                itr[s, t, j] = 1
    ntpr = itr.sum(axis=1)
    recv_cnt = np.array([sum(1 for x in entries if x[0] == e) for e in range(E)])
    aligned = np.array([seg[e][1] - seg[e][0] for e in range(E)])
    rank_base = np.array([seg[j * L][0] for j in range(R)] + [row])
    expert_start = np.array([[seg[j * L + l][0] - rank_base[j] for l in range(L)]
                             + [rank_base[j + 1] - rank_base[j]] for j in range(R)])
    src_prefix = np.array([[sum(1 for x in entries if x[0] == e and x[1] < s) for e in range(E)]
                           for s in range(R)])
    usage = np.array([[max(aligned[j * L:(j + 1) * L]), int(np.sum(recv_cnt[j * L:(j + 1) * L] > 0))]
                      for j in range(R)])
    return dict(cnt=cnt, is_token_in_rank=itr, num_tokens_per_rank=ntpr, recv_cnt=recv_cnt,
                aligned=aligned, rank_base=rank_base, expert_start=expert_start,
                src_prefix=src_prefix, dst_row=dst, recv_src=np.array(recv_src, np.int64),
                expert_usage_stats=usage)


def assert_layout_equal(lay, ref):
    for k, v in ref.items():
        got = getattr(lay, k)
        assert np.array_equal(np.asarray(got).reshape(np.shape(v)), v), k
    L = lay.E // lay.R
    assert np.array_equal(lay.expert_ids, np.tile(np.arange(L), (lay.R, 1)))


def test_exhaustive_tiny():
    # every topk pattern of R=2, T=2, K=1 over E=4 experts (with -1), and K=2 samples
    R, T, E = 2, 2, 4
    for alpha in (1, 2, 3):
        for pat in itertools.product(range(-1, E), repeat=R * T):
            topk = np.array(pat, np.int64).reshape(R, T, 1)
            lay = oracle.layout(R, T, E, 1, alpha, topk)
            assert lay.status == 0
            assert_layout_equal(lay, brute_layout(R, T, E, 1, alpha, topk))


def test_exhaustive_tiny_k2_with_duplicates():
    # K=2 over E=2 on R=2, T=2: all 3^8 patterns, duplicates included (k breaks ties)
    R, T, E, K = 2, 2, 2, 2
    for alpha in (1, 2):
        for pat in itertools.product(range(-1, E), repeat=R * T * K):
            topk = np.array(pat, np.int64).reshape(R, T, K)
            lay = oracle.layout(R, T, E, K, alpha, topk)
            assert_layout_equal(lay, brute_layout(R, T, E, K, alpha, topk))


@pytest.mark.parametrize("seed", range(40))
def test_random_small(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    L = int(rng.integers(1, 4))
    E = R * L
    K = int(rng.integers(1, min(E, 4) + 1))
    T = int(rng.integers(0, 9))
    alpha = int(rng.integers(1, 6))
    topk = rng.integers(-1, E, size=(R, T, K))
    lay = oracle.layout(R, T, E, K, alpha, topk)
    assert_layout_equal(lay, brute_layout(R, T, E, K, alpha, topk))


def check_invariants(lay, topk):
    R, T, E, K, alpha = lay.R, lay.T, lay.E, lay.K, lay.alpha
    L = E // R
    tk = topk.reshape(R * T * K)
    valid = tk >= 0
    V = int(valid.sum())
    # I1: token conservation
    assert int(lay.recv_cnt.sum()) == V
    assert int(lay.cnt.sum()) == V
    # I2: alignment
    assert np.all(lay.aligned % alpha == 0)
    assert np.all((lay.aligned - lay.recv_cnt >= 0) & (lay.aligned - lay.recv_cnt < alpha))
    # I3: starts monotone, last = rank rows, ranks back to back
    es = lay.expert_start
    assert np.all(np.diff(es, axis=1) >= 0)
    assert np.array_equal(es[:, -1], np.diff(lay.rank_base))
    assert lay.rank_base[0] == 0
    # I4: dst_row is a bijection of valid entries onto non-padding rows
    d = lay.dst_row.reshape(-1)
    assert np.all(d[~valid] == -1)
    dv = d[valid]
    assert len(np.unique(dv)) == V
    rs = lay.recv_src
    assert int((rs >= 0).sum()) == V
    n_of = np.repeat(np.arange(R * T), K)[valid]
    assert np.array_equal(rs[dv], n_of)
    # within each expert segment, sources strictly increase
    base = np.concatenate([[0], np.cumsum(lay.aligned)])
    for e in range(E):
        seg = rs[base[e]:base[e] + lay.recv_cnt[e]]
        assert np.all(np.diff(seg) > 0) or len(seg) <= 1
        assert np.all(rs[base[e] + lay.recv_cnt[e]:base[e + 1]] == -1)
        # every row of the segment belongs to a token routed to e
        assert np.all(np.any(topk.reshape(R * T, K)[seg] == e, axis=1))
    # tokens per rank = sum of is_token_in_rank
    assert np.array_equal(lay.num_tokens_per_rank, lay.is_token_in_rank.sum(axis=1))
    # per-source-rank expert counts match a histogram
    for s in range(R):
        h = np.bincount(topk[s][topk[s] >= 0].ravel(), minlength=E)
        assert np.array_equal(lay.cnt[s], h)
    # src_prefix is the exclusive cumulative sum over source ranks
    assert np.array_equal(lay.src_prefix, np.cumsum(lay.cnt, axis=0) - lay.cnt)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_invariants_scaled_workloads(idx):
    w = synth.WORKLOADS[idx]
    w = w.with_(T=min(w.T, 256))
    topk = synth.gen_topk(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    assert lay.status == 0
    check_invariants(lay, topk)


def test_workload1_matches_brute_force():
    w = synth.WORKLOADS[1]
    topk = synth.gen_topk(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    assert_layout_equal(lay, brute_layout(w.R, w.T, w.E, w.K, w.alpha, topk))


def test_zipf_workload_skew_small():
    w = synth.WORKLOADS[3].with_(T=64)
    topk = synth.gen_topk(w)
    lay = oracle.layout(w.R, w.T, w.E, w.K, w.alpha, topk)
    assert_layout_equal(lay, brute_layout(w.R, w.T, w.E, w.K, w.alpha, topk))
    # Zipf(1.2) without permutation puts the heaviest experts on rank 0
    assert lay.recv_cnt[0] == lay.recv_cnt.max()


def test_edge_cases():
    # T = 0: no rows at all
    lay = oracle.layout(2, 0, 4, 2, 4, np.zeros((2, 0, 2), np.int64))
    assert lay.rows == 0 and lay.status == 0
    # every entry -1: no rows, no token in any rank
    topk = -np.ones((2, 3, 2), np.int64)
    lay = oracle.layout(2, 3, 4, 2, 8, topk)
    assert lay.rows == 0 and np.all(lay.dst_row == -1) and lay.is_token_in_rank.sum() == 0
    # alignment larger than every count
    topk = np.array([[[0], [1]], [[1], [3]]], np.int64)
    lay = oracle.layout(2, 2, 4, 1, 16, topk)
    assert np.array_equal(lay.aligned, [16, 16, 0, 16]) and lay.rows == 48
    assert_layout_equal(lay, brute_layout(2, 2, 4, 1, 16, topk))
    # L = 1 (one expert per rank), K = 1
    topk = np.array([[[2], [0]], [[1], [2]], [[0], [-1]]], np.int64)
    lay = oracle.layout(3, 2, 3, 1, 1, topk)
    assert_layout_equal(lay, brute_layout(3, 2, 3, 1, 1, topk))


def test_bad_expert_id_and_capacity():
    topk = np.array([[[0, 7]], [[1, -3]]], np.int64)  # 7 and -3 are outside [-1, 4)
    lay = oracle.layout(2, 1, 4, 2, 1, topk)
    assert lay.status == 4
    assert lay.dst_row.reshape(-1).tolist() == [0, -1, 1, -1]
    topk = np.array([[[0, 1]], [[0, 1]]], np.int64)
    lay = oracle.layout(2, 1, 4, 2, 1, topk, recv_cap=3)
    assert lay.status == 3 and lay.rows == 4
