"""Pins of the oracle's non-expand layout (EPHandle do_expand = false, "DeepEP
overall architecture analysis": one receive row per (token, destination rank))
and of the routing forwarded with its rows, against a hand-worked example,
brute-force enumeration, the expand layout in the case where the two coincide,
invariants, and closed forms of dispatch and combine over its rows."""
import numpy as np
import pytest

import oracle
import synth
from layout_checks import check_layout_nonexpand


def run(topk, W, T, Epr, A, rcap=None):
    return oracle.layout_nonexpand(np.asarray(topk, dtype=np.int64), W, T, Epr, A, rcap)


def check(o, topk, W, T, Epr, A):
    check_layout_nonexpand(topk, W, T, Epr, A, o["rcap"], o["cnt"], o["tok_per_rank"],
                           o["psum_expert"], o["psum_rank"], o["dst_slot"], o["send_slot"],
                           o["meta"], o["num_recv"])


def test_worked_example_by_hand():
    # W=2, T=2, Epr=2 (experts 0,1 on rank 0; 2,3 on rank 1), K=2, A=1.
    #  t0 -> e0, e3 (ranks 0, 1); t1 -> e1, e0 (rank 0 twice); t2 -> e2, e3 (rank 1
    #  twice); t3 -> masked, e1 (rank 0).
    # rank 0 receives t0, t1, t3 -> rows 0, 1, 2; rank 1 receives t0, t2 -> rows 3, 4.
    # capacity = W*T*min(K, W) = 8.
    o = run([[0, 3], [1, 0], [2, 3], [-1, 1]], 2, 2, 2, 1)
    assert o["rcap"] == 8
    assert o["cnt"].tolist() == [2, 2, 1, 2]
    assert o["psum_expert"].tolist() == [0, 2, 4, 5, 7]
    assert o["tok_per_rank"].tolist() == [3, 2]
    assert o["psum_rank"].tolist() == [0, 3, 5]
    assert o["num_recv"] == 5
    assert o["dst_slot"].tolist() == [[0, 3], [1, 1], [4, 4], [-1, 2]]
    assert o["send_slot"].tolist() == [[0, 3], [1, -1], [4, -1], [2, -1]]
    m = -1
    assert o["meta"].tolist() == [
        [0, 0, 0, 3],    # row 0: t0 on rank 0
        [0, 1, 1, 1],    # row 1: t1
        [1, 1, -1, 2],   # row 2: t3 (source rank 1, local 1)
        [0, 0, 0, 3],    # row 3: t0 on rank 1
        [1, 0, 4, 4],    # row 4: t2
        [m, m, m, m], [m, m, m, m], [m, m, m, m],
    ]
    # forwarded routing: K-wide rows, the token's entries carried by the row
    w = np.array([[0.25, 0.75], [0.5, 0.5], [0.125, 0.875], [0.0, 1.0]], np.float32)
    rw = np.full((8, 2), 9.0, np.float32)
    ri = np.full((8, 2), 9, np.int32)
    oracle.forward_routing_nonexpand(np.array([[0, 3], [1, 0], [2, 3], [-1, 1]]), w,
                                     o["dst_slot"], o["send_slot"], rw, ri)
    assert ri.tolist() == [[0, -1], [1, 0], [-1, 1], [-1, 3], [2, 3], [9, 9], [9, 9], [9, 9]]
    assert rw.tolist() == [[0.25, 0.0], [0.5, 0.5], [0.0, 1.0], [0.0, 0.75], [0.125, 0.875],
                           [9, 9], [9, 9], [9, 9]]


def brute_force(topk, W, T, Epr):
    """Rank by rank, the tokens that have an expert there, in token order."""
    N = len(topk)
    K = len(topk[0]) if N else 0
    E = W * Epr
    rows = {}
    base = 0
    psum = [0]
    for r in range(W):
        toks = [t for t in range(N) if any(0 <= e < E and e // Epr == r for e in topk[t])]
        for j, t in enumerate(toks):
            rows[(t, r)] = base + j
        base += len(toks)
        psum.append(base)
    dst = [[rows[(t, topk[t][k] // Epr)] if 0 <= topk[t][k] < E else -1 for k in range(K)]
           for t in range(N)]
    send = []
    for t in range(N):
        mine = sorted(v for (tt, _), v in rows.items() if tt == t)
        send.append(mine + [-1] * (K - len(mine)))
    return psum, dst, send


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    W = int(rng.integers(1, 6))
    Epr = int(rng.integers(1, 4))
    T = int(rng.integers(1, 7))
    N = int(rng.integers(0, W * T + 1))
    K = int(rng.integers(1, 6))
    A = int(rng.choice([1, 2, 4]))
    E = W * Epr
    topk = rng.integers(-1, E, size=(N, K)).tolist()     # duplicates and masks allowed
    o = run(np.array(topk, dtype=np.int64).reshape(N, K), W, T, Epr, A)
    psum, dst, send = brute_force(topk, W, T, Epr)
    assert o["psum_rank"].tolist() == psum
    assert o["dst_slot"].tolist() == (dst if N else [])
    assert o["send_slot"].tolist() == (send if N else [])
    assert o["rcap"] == W * T * min(K, W)
    check(o, np.array(topk, dtype=np.int64).reshape(N, K), W, T, Epr, A)


@pytest.mark.parametrize("seed", range(4))
def test_equals_the_expand_layout_with_one_expert_per_rank(seed):
    # Epr = 1, A = 1 and distinct experts per token: rows per rank are rows per
    # expert, both ordered by token, so the two layouts coincide.
    rng = np.random.default_rng(seed)
    W, T, K = 8, 16, 3
    topk = np.stack([rng.permutation(W)[:K] for _ in range(W * T)]).astype(np.int64)
    topk[rng.random(topk.shape) < 0.1] = -1
    ne = run(topk, W, T, 1, 1)
    ex = oracle.layout(topk, W, T, 1, 1)
    for key in ("cnt", "tok_per_rank", "psum_rank", "dst_slot"):
        assert np.array_equal(ne[key], ex[key]), key
    assert ne["num_recv"] == ex["num_recv"]
    assert np.array_equal(ne["meta"], ex["meta"][:ne["rcap"]])
    assert np.all(ex["meta"][ne["rcap"]:] == -1)
    # send_slot holds the same rows, sorted
    want = np.sort(np.where(ex["dst_slot"] < 0, np.iinfo(np.int32).max, ex["dst_slot"]), axis=1)
    want[want == np.iinfo(np.int32).max] = -1
    assert np.array_equal(ne["send_slot"], want)


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_invariants_on_the_workloads(name):
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl, mask_frac=0.05).numpy()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, wl.alignment)
    check(o, topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, wl.alignment)
    ex = oracle.layout(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.alignment)
    assert np.array_equal(o["cnt"], ex["cnt"]) and np.array_equal(o["psum_expert"], ex["psum_expert"])
    assert np.array_equal(o["tok_per_rank"], ex["tok_per_rank"])


def test_out_of_range_ids_raise_the_error_bit():
    o = run([[0, 7], [1, -1]], 2, 1, 2, 1)
    assert o["err"] == 1
    assert o["dst_slot"].tolist() == [[0, -1], [1, -1]]
    assert o["send_slot"].tolist() == [[0, -1], [1, -1]]


@pytest.mark.parametrize("mistake", ["swap_rows", "no_dedup", "descending", "wrong_meta",
                                     "inclusive_psum"])
def test_checker_catches_planted_mistakes(mistake):
    topk = np.array([[0, 3], [1, 0], [2, 3], [-1, 1]], np.int64)
    o = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in run(topk, 2, 2, 2, 1).items()}
    if mistake == "swap_rows":
        o["send_slot"][0, 0], o["send_slot"][1, 0] = o["send_slot"][1, 0], o["send_slot"][0, 0]
    elif mistake == "no_dedup":
        o["send_slot"][1] = [1, 1]
    elif mistake == "descending":
        o["send_slot"][0] = [3, 0]
    elif mistake == "wrong_meta":
        o["meta"][4, 1] = 1
    else:
        o["psum_rank"] = np.array([3, 5, 5], np.int32)
    with pytest.raises(AssertionError):
        check(o, topk, 2, 2, 2, 1)


def test_dispatch_and_combine_over_the_rows():
    # Dispatch to send_slot puts x[t] in exactly the rows of its ranks; combining
    # those rows unweighted (identity experts) gives bf16(n_t * x[t]) with n_t <= 4
    # the number of ranks the token reached: every partial sum j * x (j <= 4, x bf16)
    # is exact in fp32, so the fold rounds once, at the end.
    wl = synth.WORKLOADS["tiny"]           # W = 4, K = 4
    topk = synth.gen_topk(wl, mask_frac=0.1).numpy()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, 1)
    x = synth.bits16(synth.gen_x(wl))
    recv = np.full((o["rcap"], wl.hidden), 0xFFFF, np.uint16)
    oracle.dispatch_bf16(x, o["send_slot"], recv)
    for t in range(wl.num_tokens):
        for s in o["send_slot"][t][o["send_slot"][t] >= 0]:
            assert np.array_equal(recv[s], x[t])
    assert np.all(recv[o["num_recv"]:] == 0xFFFF)
    out = oracle.combine(recv, o["send_slot"], None)
    n = (o["send_slot"] >= 0).sum(axis=1)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    import torch
    want = torch.from_numpy(xf * n[:, None].astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    want[n == 0] = 0                       # nothing received: the fold's +0.0
    assert set(np.unique(n)) >= {1, 2, 3, 4}
    assert np.array_equal(out, want)
    assert np.all(out[n == 0] == 0)


def test_forwarded_rows_follow_the_rank_of_each_entry():
    wl = synth.WORKLOADS["decode"]          # W = 8, Epr = 8, K = 8
    topk = synth.gen_topk(wl, mask_frac=0.05).numpy()
    w = synth.gen_weights(wl).numpy()
    Epr = wl.num_expert_per_rank
    o = run(topk, wl.world_size, wl.max_tok_per_rank, Epr, 1)
    K = wl.topk
    rw = np.full((o["rcap"], K), np.nan, np.float32)
    ri = np.full((o["rcap"], K), -7, np.int32)
    oracle.forward_routing_nonexpand(topk, w, o["dst_slot"], o["send_slot"], rw, ri)
    owner = np.searchsorted(o["psum_rank"], np.arange(o["rcap"]), side="right") - 1
    for t in range(wl.num_tokens):
        for s in o["send_slot"][t][o["send_slot"][t] >= 0]:
            mine = (topk[t] >= 0) & (topk[t] // Epr == owner[s])
            assert np.array_equal(ri[s], np.where(mine, topk[t], -1))
            assert np.array_equal(rw[s], np.where(mine, w[t], 0.0).astype(np.float32))
    R = o["num_recv"]
    assert np.all(ri[R:] == -7) and np.all(np.isnan(rw[R:]))
    # every valid entry is carried by exactly one row
    assert (ri[:R] >= 0).sum() == (topk >= 0).sum()
