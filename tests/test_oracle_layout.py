"""Pins of the oracle's layout (histogram, aligned exclusive prefix sums, slots,
recv_src_metadata) against things other than the oracle itself: a hand-worked
example, brute-force enumeration on tiny inputs, an independent stable-sort
formulation (numpy's stable argsort) and the invariants of the EPHandle fields
("DeepEP overall architecture analysis", EPHandle class listing)."""
import numpy as np
import pytest

import oracle
import synth
from layout_checks import check_layout


def run(topk, W, T, Epr, A, rcap=None):
    return oracle.layout(np.asarray(topk, dtype=np.int64), W, T, Epr, A, rcap)


def test_worked_example_by_hand():
    # W=2 ranks, T=2 tokens per rank, Epr=2 (E=4), K=2, A=2.
    #  t0 -> e1, e2 ; t1 -> e0, e1 ; t2 -> e3, e1 ; t3 -> e1, masked
    # cnt = [1, 4, 1, 1]; aligned to 2 -> [2, 4, 2, 2]; psum = [0, 2, 6, 8, 10]
    # e1's entries in flat order (0,0) (1,1) (2,1) (3,0) get rows 2, 3, 4, 5;
    # e0: (1,0) -> 0; e2: (0,1) -> 6; e3: (2,0) -> 8.
    # capacity = W*T*K + E*(A-1) = 8 + 4 = 12.
    topk = [[1, 2], [0, 1], [3, 1], [1, -1]]
    o = run(topk, 2, 2, 2, 2)
    assert o["rcap"] == 12
    assert o["cnt"].tolist() == [1, 4, 1, 1]
    assert o["psum_expert"].tolist() == [0, 2, 6, 8, 10]
    assert o["psum_rank"].tolist() == [0, 6, 10]
    assert o["tok_per_rank"].tolist() == [4, 2]
    assert o["num_recv"] == 10
    assert o["dst_slot"].tolist() == [[2, 6], [0, 3], [8, 4], [5, -1]]
    m = -1
    assert o["meta"].tolist() == [
        [0, 1, 0, 3],    # row 0: t1 (rank 0, local 1)
        [m, m, m, m],    # row 1: padding of e0
        [0, 0, 2, 6],    # row 2: t0
        [0, 1, 0, 3],    # row 3: t1
        [1, 0, 8, 4],    # row 4: t2 (rank 1, local 0)
        [1, 1, 5, -1],   # row 5: t3
        [0, 0, 2, 6],    # row 6: t0
        [m, m, m, m],    # row 7: padding of e2
        [1, 0, 8, 4],    # row 8: t2
        [m, m, m, m],    # row 9: padding of e3
        [m, m, m, m],    # rows 10, 11: beyond R
        [m, m, m, m],
    ]
    assert o["err"] == 0


def brute_force(topk, W, T, Epr, A):
    """Enumerate, expert by expert, the (t, k) entries routed to it."""
    N, K = len(topk), len(topk[0]) if topk else 0
    E = W * Epr
    slot = [[-1] * K for _ in range(N)]
    cnt = [0] * E
    base = 0
    psum = [0]
    for e in range(E):
        rows = [(t, k) for t in range(N) for k in range(K) if topk[t][k] == e]
        for j, (t, k) in enumerate(rows):
            slot[t][k] = base + j
        cnt[e] = len(rows)
        base += -(-len(rows) // A) * A
        psum.append(base)
    return cnt, psum, slot


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    W = int(rng.integers(1, 5))
    Epr = int(rng.integers(1, 5))
    T = int(rng.integers(1, 7))
    N = int(rng.integers(0, W * T + 1))
    K = int(rng.integers(1, 5))
    A = int(rng.choice([1, 2, 3, 4, 8]))
    E = W * Epr
    # duplicates and masked entries allowed
    topk = rng.integers(-1, E, size=(N, K)).tolist()
    o = run(topk if N else np.zeros((0, K)), W, T, Epr, A)
    cnt, psum, slot = brute_force(topk, W, T, Epr, A)
    assert o["cnt"].tolist() == cnt
    assert o["psum_expert"].tolist() == psum
    assert o["dst_slot"].reshape(N, K).tolist() == slot
    check_layout(np.asarray(topk, np.int64).reshape(N, K), W, T, Epr, A, o["rcap"],
                 o["cnt"], o["tok_per_rank"], o["psum_expert"], o["psum_rank"],
                 o["dst_slot"], o["meta"], o["num_recv"])


def stable_sort_slots(topk, E, A):
    """Independent formulation: a stable sort of the flat entries by expert id
    gives, for each entry, its position among all valid entries; subtracting the
    unpadded start of its expert and adding the padded start gives the slot."""
    flat = np.asarray(topk, np.int64).ravel()
    valid = (flat >= 0) & (flat < E)
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    pos = np.empty_like(order)
    pos[order] = np.arange(len(order))
    cnt = np.bincount(flat[valid], minlength=E)
    start_unpadded = np.concatenate([[0], np.cumsum(cnt)])[:-1]
    start_padded = np.concatenate([[0], np.cumsum(-(-cnt // A) * A)])[:-1]
    slot = np.full(flat.shape, -1, np.int64)
    e = flat[valid]
    slot[valid] = pos[valid] - start_unpadded[e] + start_padded[e]
    return slot.reshape(np.asarray(topk).shape)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_stable_sort_formulation_and_invariants(name):
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl).numpy()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, wl.alignment)
    assert o["rcap"] == wl.recv_capacity
    assert np.array_equal(o["dst_slot"], stable_sort_slots(topk, wl.num_experts, wl.alignment))
    check_layout(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                 wl.alignment, o["rcap"], o["cnt"], o["tok_per_rank"], o["psum_expert"],
                 o["psum_rank"], o["dst_slot"], o["meta"], o["num_recv"])
    assert o["err"] == 0


def test_masked_entries_and_out_of_range():
    wl = synth.WORKLOADS["tiny"]
    topk = synth.gen_topk(wl, mask_frac=0.3).numpy()
    assert (topk == -1).any()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, 4)
    assert o["err"] == 0
    assert np.array_equal(o["dst_slot"], stable_sort_slots(topk, wl.num_experts, 4))
    assert int(o["cnt"].sum()) == int((topk >= 0).sum())
    bad = topk.copy()
    bad[3, 1] = wl.num_experts       # out of range: skipped, error bit set
    bad[5, 0] = -7
    o2 = run(bad, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, 4)
    assert o2["err"] == 1
    assert o2["dst_slot"][3, 1] == -1 and o2["dst_slot"][5, 0] == -1


def test_empty_batch():
    o = run(np.zeros((0, 8), np.int64), 8, 16, 4, 16)
    assert o["num_recv"] == 0
    assert not o["cnt"].any() and not o["psum_expert"].any()
    assert (o["meta"] == -1).all()


def test_skewed_routing_is_skewed():
    wl = synth.WORKLOADS["skewed"]
    topk = synth.gen_topk(wl).numpy()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, wl.alignment)
    mean = o["cnt"].mean()
    assert o["cnt"].max() > 10 * mean
    # distinct experts within a token
    assert all(len(set(r)) == wl.topk for r in topk[:2000].tolist())


@pytest.mark.parametrize("mistake", ["swap_slots", "drop_padding", "meta_col", "psum_inclusive",
                                     "cnt_off_by_one"])
def test_checker_catches_planted_mistakes(mistake):
    """The invariant checker used on every implementation fails on a layout with
    a plausible mistake planted in the oracle's output."""
    wl = synth.WORKLOADS["tiny"].with_(alignment=4)
    topk = synth.gen_topk(wl).numpy()
    o = run(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank, wl.alignment)
    o = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in o.items()}
    if mistake == "swap_slots":
        e = topk[0, 0]
        t2, k2 = [(t, k) for t in range(1, wl.num_tokens) for k in range(wl.topk)
                  if topk[t, k] == e][0]
        o["dst_slot"][0, 0], o["dst_slot"][t2, k2] = o["dst_slot"][t2, k2], o["dst_slot"][0, 0]
    elif mistake == "drop_padding":
        o["psum_expert"] = np.concatenate([[0], np.cumsum(o["cnt"])]).astype(np.int32)
    elif mistake == "meta_col":
        r = o["dst_slot"][1, 0]
        o["meta"][r, 1] += 1
    elif mistake == "psum_inclusive":
        o["psum_expert"] = np.concatenate([o["psum_expert"][1:], [o["psum_expert"][-1]]])
    elif mistake == "cnt_off_by_one":
        o["cnt"][2] += 1
    with pytest.raises(AssertionError):
        check_layout(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                     wl.alignment, o["rcap"], o["cnt"], o["tok_per_rank"], o["psum_expert"],
                     o["psum_rank"], o["dst_slot"], o["meta"], o["num_recv"])
