"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bar: layout fields, slots, metadata and dispatched bf16 / e4m3 bytes and
scales are bit-exact; combine is bit-exact too, because both sides fold the K
rows in the same fixed fma order (the looser tolerance max-abs <= 1e-2 and
rel-L2 <= 1e-3 is asserted as well).  Sizes: whole-array comparison on all five
workloads.  At the prefill sizes (32768 tokens x 7168, the launch
configuration the benchmark times) the oracle runs range by range (2048 tokens
at a time, into compact buffers) so that every received row, every scale and
every combined token is still compared; properties that hold at any size
(untouched padding rows, the identity-expert round trip) are checked too.
"""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth
from layout_checks import check_layout, LAYOUT_PATHS, set_layout_path, ran_path

pytestmark = pytest.mark.gpu

FIELDS = {
    "cnt": ep.FIELD_NUM_UNALIGNED_PER_EXPERT,
    "tok_per_rank": ep.FIELD_NUM_TOKENS_PER_RANK,
    "psum_expert": ep.FIELD_PSUM_PER_EXPERT,
    "psum_rank": ep.FIELD_PSUM_PER_RANK,
    "dst_slot": ep.FIELD_DST_SLOT,
    "meta": ep.FIELD_RECV_SRC_METADATA,
}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def cfg_of(wl, dtype=None, use_weights=None):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, dtype or wl.dispatch_dtype,
                       wl.use_weights if use_weights is None else use_weights)


def oracle_layout(wl, topk):
    return oracle.layout(np.asarray(topk), wl.world_size, wl.max_tok_per_rank,
                         wl.num_expert_per_rank, wl.alignment)


def gpu_fields(h):
    torch.cuda.synchronize()
    out = {k: h.field(f).cpu().numpy() for k, f in FIELDS.items()}
    out["num_recv"] = int(h.field(ep.FIELD_NUM_RECV).cpu()[0])
    return out


def assert_layout_equal(got, ref):
    for k in list(FIELDS) + ["num_recv"]:
        assert np.array_equal(np.asarray(got[k]), np.asarray(ref[k])), k


def layout_case(wl, topk_cpu):
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk_cpu.cuda())
    got = gpu_fields(h)
    ref = oracle_layout(wl, topk_cpu.numpy())
    return h, got, ref


# ------------------------------------------------------------------- layout

@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_layout_bit_exact(name):
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl)
    h, got, ref = layout_case(wl, topk)
    assert_layout_equal(got, ref)
    check_layout(topk.numpy(), wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                 wl.alignment, wl.recv_capacity, got["cnt"], got["tok_per_rank"],
                 got["psum_expert"], got["psum_rank"], got["dst_slot"], got["meta"],
                 got["num_recv"])
    assert h.status() == 0
    # deterministic: a second run gives the same bytes
    h.layout(topk.cuda())
    again = gpu_fields(h)
    assert_layout_equal(again, ref)


EDGE = {
    # masked entries
    "masked": dict(base="decode", mask_frac=0.2),
    # ragged batch: N not a multiple of the 128-token chunk
    "ragged": dict(base="decode", num_tokens=1000),
    "one_token": dict(base="tiny", num_tokens=1),
    # generic (unspecialised) top-k and hidden, odd metadata width
    "generic_k5": dict(base="tiny", topk=5, hidden=384, alignment=3),
    "k1": dict(base="tiny", topk=1, alignment=8),
    "k16": dict(base="tiny", topk=16, num_expert_per_rank=16, alignment=16),
    # the largest expert count the library accepts (2048) with 64 ranks
    "max_experts": dict(base="tiny", world_size=64, num_expert_per_rank=32, max_tok_per_rank=64,
                        num_tokens=4096, topk=8, alignment=2),
    "big_alignment": dict(base="decode", alignment=4096),
    # one expert per rank, and a non-power-of-two experts-per-rank
    "epr1": dict(base="tiny", num_expert_per_rank=1, topk=4, alignment=2),
    "epr7": dict(base="tiny", world_size=3, num_expert_per_rank=7, max_tok_per_rank=64,
                 num_tokens=150, alignment=5),
    "zipf_hot": dict(base="skewed", num_tokens=4096),
}


def edge_wl(spec):
    spec = dict(spec)
    base = synth.WORKLOADS[spec.pop("base")]
    mask = spec.pop("mask_frac", 0.0)
    return base.with_(**spec), mask


@pytest.mark.parametrize("case", list(EDGE))
def test_layout_edge_cases(case):
    wl, mask = edge_wl(EDGE[case])
    topk = synth.gen_topk(wl, mask_frac=mask)
    h, got, ref = layout_case(wl, topk)
    assert_layout_equal(got, ref)
    assert h.status() == 0


def test_layout_all_tokens_to_one_expert():
    wl = synth.WORKLOADS["decode"].with_(topk=1, alignment=128)
    topk = torch.full((wl.num_tokens, 1), 5, dtype=torch.int64)
    h, got, ref = layout_case(wl, topk)
    assert_layout_equal(got, ref)
    assert got["cnt"][5] == wl.num_tokens


def test_layout_empty_batch():
    wl = synth.WORKLOADS["decode"].with_(alignment=16)
    h = ep.EpHandle(cfg_of(wl))
    # fill the handle with a real routing first, then an empty one must clear it
    h.layout(synth.gen_topk(wl).cuda())
    h.layout(torch.zeros((0, wl.topk), dtype=torch.int64, device="cuda"))
    got = gpu_fields(h)
    ref = oracle_layout(wl, np.zeros((0, wl.topk), np.int64))
    assert_layout_equal(got, ref)
    assert got["num_recv"] == 0 and (got["meta"] == -1).all()
    # dispatch / combine of nothing are no-ops
    h.dispatch(torch.zeros((0, wl.hidden), dtype=torch.bfloat16, device="cuda"),
               torch.zeros((1, wl.hidden), dtype=torch.bfloat16, device="cuda"))
    h.combine(torch.zeros((1, wl.hidden), dtype=torch.bfloat16, device="cuda"),
              torch.zeros((0, wl.topk), device="cuda"),
              torch.zeros((0, wl.hidden), dtype=torch.bfloat16, device="cuda"))
    assert h.status() == 0


def test_out_of_range_ids_are_skipped_and_flagged():
    wl = synth.WORKLOADS["tiny"]
    topk = synth.gen_topk(wl)
    topk[3, 1] = wl.num_experts
    topk[7, 0] = -5
    topk[9, 2] = -1
    h, got, ref = layout_case(wl, topk)
    assert ref["err"] == 1
    assert_layout_equal(got, ref)
    assert h.status() == ep.ERR_BAD_EXPERT
    assert h.status() == 0  # read clears it


# ----------------------------------------------------------------- dispatch

CANARY16 = -1  # 0xFFFF as int16, a bf16 NaN pattern


def dispatch_bf16_case(wl, mask=0.0):
    case = synth.make_case(wl, device="cuda", mask_frac=mask)
    h = ep.EpHandle(cfg_of(wl, "bf16"))
    h.layout(case["topk_idx"].cuda())
    recv = torch.full((wl.recv_capacity, wl.hidden), CANARY16, dtype=torch.int16,
                      device="cuda").view(torch.bfloat16)
    h.dispatch(case["x"], recv)
    torch.cuda.synchronize()
    ref = oracle_layout(wl, case["topk_idx"].numpy())
    return h, case, recv, ref


@pytest.mark.parametrize("name,mask", [("tiny", 0.0), ("tiny", 0.25), ("decode", 0.0),
                                       ("skewed", 0.0)])
def test_dispatch_bf16_whole_buffer(name, mask):
    wl = synth.WORKLOADS[name]
    h, case, recv, ref = dispatch_bf16_case(wl, mask)
    want = np.full((wl.recv_capacity, wl.hidden), 0xFFFF, np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], want)
    assert np.array_equal(synth.bits16(recv), want)
    assert h.status() == 0


@pytest.mark.parametrize("case_name", ["generic_k5", "k16", "ragged", "one_token"])
def test_dispatch_bf16_edge(case_name):
    wl, mask = edge_wl(EDGE[case_name])
    h, case, recv, ref = dispatch_bf16_case(wl, mask)
    want = np.full((wl.recv_capacity, wl.hidden), 0xFFFF, np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], want)
    assert np.array_equal(synth.bits16(recv), want)


def compact_slots(dst_slot_sel):
    """Slots renumbered 0..n*K-1 in (t, k) order, -1 kept."""
    s = np.arange(dst_slot_sel.size, dtype=np.int32).reshape(dst_slot_sel.shape)
    return np.where(dst_slot_sel >= 0, s, -1).astype(np.int32)


def padding_rows(ref):
    return np.flatnonzero(ref["meta"][:, 0] == -1)


RANGE = 2048   # tokens per oracle pass in the whole-buffer prefill comparisons


def token_ranges(n):
    return [(a, min(n, a + RANGE)) for a in range(0, n, RANGE)]


def test_dispatch_bf16_prefill_whole():
    """Every received row of the 32768-token prefill dispatch against the oracle,
    range by range: the oracle writes the range's rows into a compact buffer
    (slots renumbered in (t, k) order) and the GPU rows at the range's real slots
    must hold the same bytes.  Padding rows keep their canary."""
    wl = synth.WORKLOADS["prefill_bf16"]
    h, case, recv, ref = dispatch_bf16_case(wl)
    assert_layout_equal(gpu_fields(h), ref)
    xb = synth.bits16(case["x"])
    covered = 0
    for a, b in token_ranges(wl.num_tokens):
        ds = ref["dst_slot"][a:b]
        want = np.zeros((ds.size, wl.hidden), np.uint16)
        oracle.dispatch_bf16(xb[a:b], compact_slots(ds), want)
        rows = torch.from_numpy(ds.reshape(-1).astype(np.int64)).cuda()
        got = recv.view(torch.int16)[rows]
        assert torch.equal(got, torch.from_numpy(want.view(np.int16)).cuda()), (a, b)
        covered += ds.size
    # every received row was compared: one per (token, k), none left out
    assert covered == wl.num_tokens * wl.topk == int((ref["meta"][:, 0] >= 0).sum())
    pad = torch.from_numpy(padding_rows(ref)).cuda()
    assert bool((recv.view(torch.int16)[pad] == CANARY16).all())
    assert h.status() == 0


def fp8_case(wl, mask=0.0):
    case = synth.make_case(wl, device="cuda", mask_frac=mask)
    h = ep.EpHandle(cfg_of(wl, "fp8"))
    h.layout(case["topk_idx"].cuda())
    G = wl.hidden // 128
    rq = torch.full((wl.recv_capacity, wl.hidden), 0xAB, dtype=torch.uint8, device="cuda")
    rs = torch.full((wl.recv_capacity, G), -7.0, dtype=torch.float32, device="cuda")
    h.dispatch(case["x"], rq, rs)
    torch.cuda.synchronize()
    ref = oracle_layout(wl, case["topk_idx"].numpy())
    return h, case, rq, rs, ref


@pytest.mark.parametrize("name,over", [("tiny", {}), ("decode", {}), ("tiny", {"hidden": 384}),
                                       ("tiny", {"topk": 5, "hidden": 640, "alignment": 4}),
                                       ("skewed", {"num_tokens": 2048})])
def test_dispatch_fp8_whole_buffer(name, over):
    wl = synth.WORKLOADS[name].with_(dispatch_dtype="fp8", **over)
    h, case, rq, rs, ref = fp8_case(wl, mask=0.1 if name == "tiny" else 0.0)
    G = wl.hidden // 128
    q = np.full((wl.recv_capacity, wl.hidden), 0xAB, np.uint8)
    s = np.full((wl.recv_capacity, G), -7.0, np.float32)
    oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], q, s)
    assert np.array_equal(rq.cpu().numpy(), q)
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert h.status() == 0


def test_dispatch_fp8_special_values():
    """Groups that are all zero, contain -0.0, a power-of-two amax, tiny and huge
    values: bytes and scales must match the oracle's encoder exactly."""
    wl = synth.WORKLOADS["tiny"].with_(dispatch_dtype="fp8", hidden=1024)
    topk = synth.gen_topk(wl)
    x = synth.gen_bf16_normal(wl.num_tokens, wl.hidden, seed=5).float()
    x[0, :128] = 0.0
    x[1, :128] = 0.0
    x[1, 5] = -0.0
    x[1, 6] = 2.0
    x[2, 128:256] *= 1e-30
    x[3, 256:384] *= 1e30
    x[4, 384:512] = torch.linspace(-448, 448, 128)
    x[5, 512:640] = -0.0
    xb = x.to(torch.bfloat16).cuda()
    h = ep.EpHandle(cfg_of(wl, "fp8"))
    h.layout(topk.cuda())
    rq = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.uint8, device="cuda")
    rs = torch.zeros((wl.recv_capacity, 8), dtype=torch.float32, device="cuda")
    h.dispatch(xb, rq, rs)
    ref = oracle_layout(wl, topk.numpy())
    q = np.zeros((wl.recv_capacity, wl.hidden), np.uint8)
    s = np.zeros((wl.recv_capacity, 8), np.float32)
    oracle.dispatch_fp8(synth.bits16(xb), ref["dst_slot"], q, s)
    assert np.array_equal(rq.cpu().numpy(), q)
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_dispatch_fp8_prefill_whole():
    """Every received e4m3 row and its 56 scales of the 32768-token prefill FP8
    dispatch against the oracle, range by range; padding rows untouched."""
    wl = synth.WORKLOADS["prefill_fp8"]
    h, case, rq, rs, ref = fp8_case(wl)
    xb = synth.bits16(case["x"])
    G = wl.hidden // 128
    for a, b in token_ranges(wl.num_tokens):
        ds = ref["dst_slot"][a:b]
        q = np.zeros((ds.size, wl.hidden), np.uint8)
        s = np.zeros((ds.size, G), np.float32)
        oracle.dispatch_fp8(xb[a:b], compact_slots(ds), q, s)
        rows = torch.from_numpy(ds.reshape(-1).astype(np.int64)).cuda()
        assert torch.equal(rq[rows], torch.from_numpy(q).cuda()), (a, b)
        assert torch.equal(rs[rows].view(torch.int32), torch.from_numpy(s.view(np.int32)).cuda()), (a, b)
    pad = torch.from_numpy(padding_rows(ref)).cuda()
    assert bool((rq[pad] == 0xAB).all()) and bool((rs[pad] == -7.0).all())
    assert h.status() == 0


# ------------------------------------------------------------------ combine

def combine_case(wl, use_weights=True, mask=0.0):
    topk = synth.gen_topk(wl, mask_frac=mask)
    ref = oracle_layout(wl, topk.numpy())
    valid = ref["meta"][:, 0] >= 0
    y = synth.gen_y(wl, valid_rows=valid, device="cuda")   # padding rows are NaN
    w = synth.gen_weights(wl)
    h = ep.EpHandle(cfg_of(wl, use_weights=use_weights))
    h.layout(topk.cuda())
    out = torch.full((wl.num_tokens, wl.hidden), CANARY16, dtype=torch.int16,
                     device="cuda").view(torch.bfloat16)
    h.combine(y, w.cuda() if use_weights else None, out)
    torch.cuda.synchronize()
    return h, ref, y, w, out


def assert_combine_close(got_bits, want_bits):
    assert np.array_equal(got_bits, want_bits)  # same fma order: bit-exact
    g = torch.from_numpy(got_bits.view(np.int16)).view(torch.bfloat16).double()
    r = torch.from_numpy(want_bits.view(np.int16)).view(torch.bfloat16).double()
    assert torch.isfinite(g).all()
    assert (g - r).abs().max() <= 1e-2
    assert (g - r).norm() <= 1e-3 * r.norm() + 1e-30


@pytest.mark.parametrize("name,use_w,mask", [("tiny", True, 0.0), ("tiny", False, 0.2),
                                             ("decode", True, 0.0), ("decode", False, 0.0),
                                             ("skewed", True, 0.0)])
def test_combine_whole(name, use_w, mask):
    wl = synth.WORKLOADS[name]
    h, ref, y, w, out = combine_case(wl, use_w, mask)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], w.numpy() if use_w else None)
    assert_combine_close(synth.bits16(out), want)


@pytest.mark.parametrize("case_name", ["generic_k5", "k16", "k1", "ragged"])
def test_combine_edge(case_name):
    wl, mask = edge_wl(EDGE[case_name])
    h, ref, y, w, out = combine_case(wl, True, mask)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], w.numpy())
    assert_combine_close(synth.bits16(out), want)


@pytest.mark.parametrize("name", ["prefill_bf16", "prefill_fp8"])
def test_combine_prefill_whole(name):
    """Every token of the 32768-token prefill combine against the oracle, range by
    range (the range's expert rows gathered into a compact buffer for the
    oracle); bit-exact, and within max-abs 1e-2 and relative L2 1e-3."""
    wl = synth.WORKLOADS[name]
    h, ref, y, w, out = combine_case(wl)
    wn = w.numpy()
    for a, b in token_ranges(wl.num_tokens):
        ds = ref["dst_slot"][a:b]
        rows = torch.from_numpy(ds.reshape(-1).astype(np.int64)).cuda()
        want = oracle.combine(synth.bits16(y[rows]), compact_slots(ds), wn[a:b])
        assert_combine_close(synth.bits16(out[a:b]), want)
    assert bool(torch.isfinite(out.float()).all())   # no padding (NaN) row was read


def test_identity_round_trip_prefill():
    """dispatch -> identity experts -> combine with unit weights gives K*x
    exactly, at full prefill size ("MORI JIT v2" §4: the identity-expert step)."""
    wl = synth.WORKLOADS["prefill_bf16"].with_(use_weights=False)
    case = synth.make_case(wl, device="cuda")
    h = ep.EpHandle(cfg_of(wl))
    h.layout(case["topk_idx"].cuda())
    recv = torch.empty((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    h.dispatch(case["x"], recv)
    out = torch.empty_like(case["x"])
    h.combine(recv, None, out)
    want = (case["x"].float() * wl.topk).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("path,tma", [(p, False) for p in LAYOUT_PATHS] + [("cluster", True)])
def test_graph_capture_replay(path, tma, monkeypatch):
    """layout -> dispatch -> identity expert -> combine (and an FP8 dispatch on
    the same layout) captured once in a CUDA graph and replayed with new
    routings written into the same input buffers ("MORI JIT v2" §4: the step
    must replay correctly, no host-side state frozen).  The kernels after the
    first are launched with programmatic stream serialisation, so each replay
    also checks that no kernel reads a predecessor's output before it is
    complete, nor a stale copy of the previous replay's.  tma: the bf16
    dispatch and the combine are the TMA-staged variants (mbarriers in the
    captured kernels)."""
    set_layout_path(monkeypatch, path)
    if tma:
        monkeypatch.setenv("EP_GB300_DISPATCH_TMA", "1")
        monkeypatch.setenv("EP_GB300_COMBINE_TMA", "1")
    wl = synth.WORKLOADS["decode"]
    h = ep.EpHandle(cfg_of(wl))
    h8 = ep.EpHandle(cfg_of(wl, "fp8"), layout_of=h)
    topk_buf = torch.zeros((wl.num_tokens, wl.topk), dtype=torch.int64, device="cuda")
    x_buf = torch.zeros((wl.num_tokens, wl.hidden), dtype=torch.bfloat16, device="cuda")
    w_buf = torch.zeros((wl.num_tokens, wl.topk), dtype=torch.float32, device="cuda")
    recv = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    rq = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.uint8, device="cuda")
    rs = torch.zeros((wl.recv_capacity, wl.hidden // 128), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x_buf)
    s = torch.cuda.Stream()
    first = synth.make_case(wl, device="cuda")
    topk_buf.copy_(first["topk_idx"])
    h.layout(topk_buf)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h.layout(topk_buf, stream=s)
        h.dispatch(x_buf, recv, stream=s)
        h.combine(recv, w_buf, out, stream=s)
        h8.dispatch(x_buf, rq, rs, stream=s)
    assert ran_path(h.variant(0)) == path, h.variant(0)
    assert ("tma" in h.variant(1) and "tma" in h.variant(2)) == tma, (h.variant(1), h.variant(2))
    for seed in range(4):
        c = synth.make_case(wl.with_(seed=0x1000 + seed), device="cuda")
        topk_buf.copy_(c["topk_idx"])
        x_buf.copy_(c["x"])
        w_buf.copy_(c["topk_weights"])
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_layout(wl, c["topk_idx"].numpy())
        assert np.array_equal(h.field(ep.FIELD_DST_SLOT).cpu().numpy(), ref["dst_slot"])
        rx = np.zeros((wl.recv_capacity, wl.hidden), np.uint16)
        xb = synth.bits16(c["x"])
        oracle.dispatch_bf16(xb, ref["dst_slot"], rx)
        real = ref["meta"][:, 0] >= 0
        assert np.array_equal(synth.bits16(recv)[real], rx[real]), seed
        want = oracle.combine(rx, ref["dst_slot"], c["topk_weights"].numpy())
        assert np.array_equal(synth.bits16(out), want), seed
        q = np.zeros((wl.recv_capacity, wl.hidden), np.uint8)
        sc = np.zeros((wl.recv_capacity, wl.hidden // 128), np.float32)
        oracle.dispatch_fp8(xb, ref["dst_slot"], q, sc)
        assert np.array_equal(rq.cpu().numpy()[real], q[real]), seed
        assert np.array_equal(rs.cpu().numpy().view(np.uint32)[real], sc.view(np.uint32)[real]), seed
    assert h.status() == 0


@pytest.mark.parametrize("name", ["decode", "skewed"])
def test_back_to_back_steps_without_synchronisation(name):
    """Several steps enqueued back to back on one stream, each with its own
    routing and activations in its own buffers but sharing the handle and the
    receive buffer: every step's combine must see its own step's rows."""
    wl = synth.WORKLOADS[name]
    h = ep.EpHandle(cfg_of(wl))
    s = torch.cuda.Stream()
    recv = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    cases, outs = [], []
    for seed in range(3):
        c = synth.make_case(wl.with_(seed=0x2000 + seed), device="cuda")
        cases.append((c, c["topk_idx"].cuda(), c["topk_weights"].cuda()))
        outs.append(torch.zeros_like(c["x"]))
    torch.cuda.synchronize()
    for (c, topk, w), out in zip(cases, outs):
        h.layout(topk, stream=s)
        h.dispatch(c["x"], recv, stream=s)
        h.combine(recv, w, out, stream=s)
    s.synchronize()
    for (c, _, _), out in zip(cases, outs):
        ref = oracle_layout(wl, c["topk_idx"].numpy())
        rx = np.zeros((wl.recv_capacity, wl.hidden), np.uint16)
        oracle.dispatch_bf16(synth.bits16(c["x"]), ref["dst_slot"], rx)
        want = oracle.combine(rx, ref["dst_slot"], c["topk_weights"].numpy())
        assert np.array_equal(synth.bits16(out), want)
    assert h.status() == 0


def test_variant_names_carry_the_shape(monkeypatch):
    wl = synth.WORKLOADS["prefill_fp8"]
    h = ep.EpHandle(cfg_of(wl))
    assert h.variant(0) == "ep_layout_k8"
    assert h.variant(1) == "ep_dispatch_fp8_h7168_k8"
    assert h.variant(2) == "ep_combine_w_h7168_k8"
    monkeypatch.setenv("EP_GB300_JIT", "0")      # no run-time specialisation
    g = ep.EpHandle(ep.make_cfg(2, 384, 8, 3, 5, 1, "bf16", False))
    assert g.variant(1) == "ep_dispatch_bf16_generic"
    assert g.variant(2) == "ep_combine_generic"
    assert g.variant(0) == "ep_layout_generic"


def test_misaligned_buffers_are_rejected():
    wl = synth.WORKLOADS["tiny"]
    h = ep.EpHandle(cfg_of(wl))
    h.layout(synth.gen_topk(wl).cuda())
    x = torch.zeros(wl.num_tokens * wl.hidden + 8, dtype=torch.bfloat16, device="cuda")
    recv = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EpError) as e:
        h.dispatch(x[1:1 + wl.num_tokens * wl.hidden], recv)
    assert e.value.code == ep.EP_EINVAL


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_sixteen_byte_aligned_buffers_take_the_16_byte_path(name):
    """Buffers that are 16- but not 32-byte aligned are served with 16-byte
    accesses; results are the same bytes."""
    wl = synth.WORKLOADS[name]
    case = synth.make_case(wl, device="cuda")
    H, R, N = wl.hidden, wl.recv_capacity, wl.num_tokens
    ref = oracle_layout(wl, case["topk_idx"].numpy())

    def off16(shape, dtype, fill=0):
        n = int(np.prod(shape))
        per = 16 // torch.tensor([], dtype=dtype).element_size()
        base = torch.full((n + 2 * per,), fill, dtype=dtype, device="cuda")
        t = base[per:per + n].view(shape)
        assert t.data_ptr() % 32 == 16
        return t

    x = off16((N, H), torch.bfloat16)
    x.copy_(case["x"])
    # bf16 dispatch + combine
    h = ep.EpHandle(cfg_of(wl, "bf16"))
    h.layout(case["topk_idx"].cuda())
    recv = off16((R, H), torch.bfloat16)
    h.dispatch(x, recv)
    out = off16((N, H), torch.bfloat16)
    h.combine(recv, case["topk_weights"].cuda(), out)
    torch.cuda.synchronize()
    rx = np.zeros((R, H), np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], rx)
    assert np.array_equal(synth.bits16(recv), rx)
    assert np.array_equal(synth.bits16(out),
                          oracle.combine(rx, ref["dst_slot"], case["topk_weights"].numpy()))
    # FP8 dispatch from a 16-byte-aligned x
    h8 = ep.EpHandle(cfg_of(wl, "fp8"))
    h8.layout(case["topk_idx"].cuda())
    rq = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
    rs = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
    h8.dispatch(x, rq, rs)
    torch.cuda.synchronize()
    q = np.zeros((R, H), np.uint8)
    s = np.zeros((R, H // 128), np.float32)
    oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], q, s)
    assert np.array_equal(rq.cpu().numpy(), q)
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), s.view(np.uint32))


# Small batches run the single-launch cluster layout; EP_GB300_LAYOUT_CLUSTER=0
# (read when the handle is built) forces the three-launch path.  Both must give
# the oracle's bytes.
SMALL = {
    "tiny": dict(base="tiny"),
    "decode_masked": dict(base="decode", mask_frac=0.2),
    "ragged_1000": dict(base="decode", num_tokens=1000),
    "two_ranges_1500": dict(base="decode", max_tok_per_rank=256, num_tokens=1500),
    "full_2048": dict(base="decode", max_tok_per_rank=256, num_tokens=2048),
    "generic_k5": dict(base="tiny", topk=5, hidden=384, alignment=3),
    "align16": dict(base="decode", alignment=16),
    "w64": dict(base="tiny", world_size=64, num_expert_per_rank=4, max_tok_per_rank=16,
                num_tokens=1024, topk=8),
    "epr7": dict(base="tiny", world_size=3, num_expert_per_rank=7, max_tok_per_rank=64,
                 num_tokens=150, alignment=5),
    # more experts than one warp scans (600): the block-wide scans
    "experts_600": dict(base="decode", num_expert_per_rank=75, max_tok_per_rank=256,
                        num_tokens=2000, alignment=4),
}


@pytest.mark.parametrize("path", LAYOUT_PATHS)
@pytest.mark.parametrize("case", list(SMALL))
def test_small_batch_layout_both_paths(case, path, monkeypatch):
    set_layout_path(monkeypatch, path)
    wl, mask = edge_wl(SMALL[case])
    topk = synth.gen_topk(wl, mask_frac=mask)
    h, got, ref = layout_case(wl, topk)
    assert_layout_equal(got, ref)
    assert h.status() == 0
    assert ran_path(h.variant(0)) == path, h.variant(0)
    # a second, different routing on the same handle
    topk2 = synth.gen_topk(wl.with_(seed=wl.seed + 1), mask_frac=0.1)
    h.layout(topk2.cuda())
    assert_layout_equal(gpu_fields(h), oracle_layout(wl, topk2.numpy()))


def test_layout_multi_million_tokens():
    # 2^22 tokens over 64 ranks: 32768 chunks, so each spine lane scans a run of
    # 1024 chunks (the loop path), and receive rows exceed 2^23
    wl = synth.WORKLOADS["tiny"].with_(world_size=64, max_tok_per_rank=65536,
                                       num_tokens=1 << 22, num_expert_per_rank=2, topk=2,
                                       alignment=4)
    g = torch.Generator().manual_seed(11)
    topk = torch.randint(-1, wl.num_experts, (wl.num_tokens, wl.topk), generator=g)
    h, got, ref = layout_case(wl, topk)
    assert_layout_equal(got, ref)
    assert got["num_recv"] > 1 << 22
    assert h.status() == 0


@pytest.mark.parametrize("jit", ["1", "0"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_largest_hidden(dtype, jit, monkeypatch):
    # hidden 32768 (64 KB bf16 rows, the largest the library accepts), a ragged
    # batch; the shape is outside the compiled table, so it runs the run-time
    # specialisation or, with it switched off, the generic kernels
    monkeypatch.setenv("EP_GB300_JIT", jit)
    wl = synth.WORKLOADS["tiny"].with_(hidden=32768, num_tokens=96, dispatch_dtype=dtype)
    case = synth.make_case(wl, device="cuda", mask_frac=0.1)
    topk, w = case["topk_idx"], case["topk_weights"]
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    ref = oracle_layout(wl, topk.numpy())
    R, H = wl.recv_capacity, wl.hidden
    if dtype == "fp8":
        recv = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
        h.dispatch(case["x"], recv, scales)
        rq = np.zeros((R, H), np.uint8)
        rs = np.zeros((R, H // 128), np.float32)
        oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], rq, rs)
        torch.cuda.synchronize()
        assert np.array_equal(recv.cpu().numpy(), rq)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
        y = synth.gen_y(wl, valid_rows=ref["meta"][:, 0] >= 0, device="cuda")
    else:
        y = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
        h.dispatch(case["x"], y)
        rx = np.zeros((R, H), np.uint16)
        oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], rx)
        torch.cuda.synchronize()
        assert np.array_equal(synth.bits16(y), rx)
    out = torch.empty((wl.num_tokens, H), dtype=torch.bfloat16, device="cuda")
    h.combine(y, w.cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bits16(out), oracle.combine(synth.bits16(y), ref["dst_slot"],
                                                            w.numpy()))
    assert h.status() == 0
    assert ("_generic" in h.variant(1)) == (jit == "0")
