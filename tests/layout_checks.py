"""Invariant checks of a layout (any implementation), written from the
definitions of the EPHandle fields in "DeepEP overall architecture analysis"
(EPHandle class listing) and the readings stated in the oracle header.

check_layout raises AssertionError naming the first violated property.
"""
import numpy as np


def check_layout(topk_idx, W, T, Epr, A, rcap, cnt, tok_per_rank, psum_expert,
                 psum_rank, dst_slot, meta, num_recv):
    topk_idx = np.asarray(topk_idx, dtype=np.int64)
    N, K = topk_idx.shape
    E = W * Epr
    valid = (topk_idx >= 0) & (topk_idx < E)
    # counts: every valid (t, k) counted once under its expert
    exp_cnt = np.bincount(topk_idx[valid].ravel(), minlength=E)
    assert np.array_equal(np.asarray(cnt), exp_cnt), "cnt != histogram of topk_idx"
    assert int(np.sum(cnt)) == int(valid.sum()), "sum(cnt) != number of valid entries"
    # distinct tokens per rank
    ranks = np.where(valid, topk_idx // Epr, -1)
    exp_tpr = np.array([(ranks == r).any(axis=1).sum() for r in range(W)], dtype=np.int64)
    assert np.array_equal(np.asarray(tok_per_rank), exp_tpr), "tok_per_rank wrong"
    # exclusive aligned prefix sum
    psum_expert = np.asarray(psum_expert, dtype=np.int64)
    assert psum_expert.shape == (E + 1,) and psum_expert[0] == 0, "psum_expert shape / start"
    d = np.diff(psum_expert)
    assert np.all(d % A == 0), "segment not a multiple of the alignment"
    assert np.all(d >= exp_cnt) and np.all(d < exp_cnt + A), "segment is not align(cnt)"
    assert int(num_recv) == int(psum_expert[E]), "num_recv != psum_expert[E]"
    assert int(num_recv) <= rcap, "receive rows exceed capacity"
    assert np.array_equal(np.asarray(psum_rank), psum_expert[np.arange(W + 1) * Epr]), \
        "psum_rank != psum_expert at rank boundaries"
    # slots: inside the expert's segment, injective, stable in flat order
    dst_slot = np.asarray(dst_slot, dtype=np.int64)
    assert np.all(dst_slot[~valid] == -1), "skipped entry has a slot"
    e = topk_idx[valid]
    s = dst_slot[valid]
    assert np.all(s >= psum_expert[e]) and np.all(s < psum_expert[e] + exp_cnt[e]), \
        "slot outside its expert's filled segment"
    assert len(np.unique(s)) == len(s), "two entries share a slot"
    flat = np.flatnonzero(valid.ravel())       # valid entries in row-major order
    ev = topk_idx.ravel()[flat]
    sv = dst_slot.ravel()[flat]
    for ex in np.unique(ev):
        ss = sv[ev == ex]
        assert np.all(np.diff(ss) == 1), "rows of an expert not in flat (t,k) order"
    # recv_src_metadata is the inverse of dst_slot, -1 elsewhere
    meta = np.asarray(meta, dtype=np.int64)
    assert meta.shape == (rcap, K + 2), "meta shape"
    exp_meta = np.full((rcap, K + 2), -1, dtype=np.int64)
    t_idx, k_idx = np.nonzero(valid)
    rows = dst_slot[t_idx, k_idx]
    exp_meta[rows, 0] = t_idx // T
    exp_meta[rows, 1] = t_idx % T
    exp_meta[rows, 2:] = dst_slot[t_idx]
    assert np.array_equal(meta, exp_meta), "recv_src_metadata is not the inverse of dst_slot"


def check_layout_nonexpand(topk_idx, W, T, Epr, A, rcap, cnt, tok_per_rank, psum_expert,
                           psum_rank, dst_slot, send_slot, meta, num_recv):
    """Invariants of the non-expand layout (EPHandle do_expand = false): one
    receive row per (token, destination rank); rank r owns rows
    [psum_rank[r], psum_rank[r+1]) holding its tokens once each in ascending
    token order; send_slot lists a token's rows in ascending order."""
    topk_idx = np.asarray(topk_idx, dtype=np.int64)
    N, K = topk_idx.shape
    E = W * Epr
    valid = (topk_idx >= 0) & (topk_idx < E)
    exp_cnt = np.bincount(topk_idx[valid].ravel(), minlength=E)
    assert np.array_equal(np.asarray(cnt), exp_cnt), "cnt != histogram of topk_idx"
    psum_expert = np.asarray(psum_expert, dtype=np.int64)
    d = np.diff(psum_expert)
    assert psum_expert[0] == 0 and np.all(d % A == 0) and np.all(d >= exp_cnt) \
        and np.all(d < exp_cnt + A), "psum_expert is not the aligned prefix of cnt"
    ranks = np.where(valid, topk_idx // Epr, -1)
    touch = np.stack([(ranks == r).any(axis=1) for r in range(W)], axis=1) if N else \
        np.zeros((0, W), bool)
    exp_tpr = touch.sum(axis=0)
    assert np.array_equal(np.asarray(tok_per_rank), exp_tpr), "tok_per_rank wrong"
    psum_rank = np.asarray(psum_rank, dtype=np.int64)
    assert psum_rank.shape == (W + 1,) and psum_rank[0] == 0, "psum_rank shape / start"
    assert np.array_equal(np.diff(psum_rank), exp_tpr), "psum_rank is not the prefix of tok_per_rank"
    assert int(num_recv) == int(psum_rank[W]) <= rcap, "num_recv != psum_rank[W] or above capacity"
    dst_slot = np.asarray(dst_slot, dtype=np.int64)
    send_slot = np.asarray(send_slot, dtype=np.int64)
    assert np.all(dst_slot[~valid] == -1), "skipped entry has a row"
    # a token's rows: one per touched rank, ascending, inside that rank's segment
    nrow = touch.sum(axis=1)
    for t in range(N):
        ss = send_slot[t]
        n = int(nrow[t])
        assert np.all(ss[n:] == -1) and np.all(ss[:n] >= 0), "send_slot not rows then -1"
        assert np.all(np.diff(ss[:n]) > 0), "send_slot not ascending"
        owner = np.searchsorted(psum_rank, ss[:n], side="right") - 1
        assert np.array_equal(owner, np.flatnonzero(touch[t])), "rows not on the token's ranks"
        for k in range(K):
            if valid[t, k]:
                j = int(np.flatnonzero(np.flatnonzero(touch[t]) == ranks[t, k])[0])
                assert dst_slot[t, k] == ss[j], "dst_slot is not the row of its rank"
    # rows of a rank in ascending token order, every row used once
    rows = send_slot[send_slot >= 0]
    assert len(np.unique(rows)) == len(rows) == int(num_recv), "rows not a bijection onto [0, R)"
    for r in range(W):
        toks = np.flatnonzero(touch[:, r])
        got = [send_slot[t][int(np.sum(touch[t, :r]))] for t in toks]
        assert np.array_equal(got, psum_rank[r] + np.arange(len(toks))), \
            "rank segment not in ascending token order"
    meta = np.asarray(meta, dtype=np.int64)
    assert meta.shape == (rcap, K + 2), "meta shape"
    exp_meta = np.full((rcap, K + 2), -1, dtype=np.int64)
    for t in range(N):
        for s in send_slot[t][send_slot[t] >= 0]:
            exp_meta[s, 0], exp_meta[s, 1] = t // T, t % T
            exp_meta[s, 2:] = dst_slot[t]
    assert np.array_equal(meta, exp_meta), "recv_src_metadata is not the inverse of send_slot"


# Layout kernels a handle may run (read from the environment when the handle is
# built): the single-launch cluster kernel (small batches), the single-launch
# fused kernel (a cooperative grid) and the three launches count / spine /
# slots.  Each path's tag in the handle's layout variant name.
LAYOUT_PATHS = ("cluster", "fused", "launches")
PATH_TAG = {"cluster": "_cluster_", "fused": "_fused_", "launches": None}


def set_layout_path(monkeypatch, path):
    """Make handles built after this call run `path` where it applies (the
    cluster and fused kernels fall back to the three launches beyond their
    limits)."""
    monkeypatch.setenv("EP_GB300_LAYOUT_CLUSTER", "1" if path == "cluster" else "0")
    monkeypatch.setenv("EP_GB300_LAYOUT_FUSED", "1" if path == "fused" else "0")


def ran_path(variant):
    """The layout path a handle's last layout ran, from its variant name."""
    for p, tag in PATH_TAG.items():
        if tag and tag in variant:
            return p
    return "launches"
