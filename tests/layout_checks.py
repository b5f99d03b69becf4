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
