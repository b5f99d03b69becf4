"""The single-launch fused layout (a cooperative grid with one grid barrier)
against the CPU oracle, bit for bit.

The fused kernel counts each token range, publishes the range's column totals
as a row of 16-bit counts and as atomic sums per superchunk of 16 ranges,
meets every other CTA at one bounded grid barrier, and then writes slots and
metadata from what it reads back.  The cases below reach: several
superchunks and a ragged last one, one range, each tokens-per-CTA setting,
the largest expert count, odd metadata widths, masked and out-of-range ids,
the expand and non-expand layouts, and many launches in a row on one handle
with changing batch sizes (the barrier state and the parity-buffered sums
carry over from launch to launch).  A wait limit of 0 makes the barrier give
up: the kernel reports device error value 2 (bit 1) and the context stays
usable.
"""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth
from layout_checks import check_layout, set_layout_path, ran_path

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


@pytest.fixture
def fused(monkeypatch):
    set_layout_path(monkeypatch, "fused")
    return monkeypatch


def cfg_of(wl, no_expand=False):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, wl.dispatch_dtype,
                       False if no_expand else wl.use_weights, no_expand=no_expand)


def ref_layout(wl, topk, no_expand=False):
    f = oracle.layout_nonexpand if no_expand else oracle.layout
    return f(np.asarray(topk), wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
             wl.alignment)


def gpu_fields(h):
    torch.cuda.synchronize()
    out = {k: h.field(f).cpu().numpy() for k, f in FIELDS.items()}
    out["num_recv"] = int(h.field(ep.FIELD_NUM_RECV).cpu()[0])
    return out


def assert_layout_equal(got, ref, what=""):
    for k in list(FIELDS) + ["num_recv"]:
        assert np.array_equal(np.asarray(got[k]), np.asarray(ref[k])), (what, k)


def run(wl, topk, no_expand=False, expect="fused"):
    h = ep.EpHandle(cfg_of(wl, no_expand))
    h.layout(topk.cuda())
    got = gpu_fields(h)
    if expect:
        assert ran_path(h.variant(0)) == expect, h.variant(0)
    assert_layout_equal(got, ref_layout(wl, topk.numpy(), no_expand), wl.name)
    return h, got


# every workload; prefill at 128, 224 and 256 tokens per CTA (256, 147 and 128
# ranges), the smaller ones also at 64 (many ranges: several superchunks) and at
# range sizes that are not powers of two
CASES = [(n, t) for n in ("tiny", "decode", "skewed") for t in (64, 96, 128, 160, 256)] + \
        [(n, t) for n in ("prefill_bf16", "prefill_fp8") for t in (128, 224, 256)]


@pytest.mark.parametrize("name,tpb", CASES)
def test_fused_layout_bit_exact(name, tpb, fused):
    fused.setenv("EP_GB300_LAYOUT_FUSED_TPB", str(tpb))
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl)
    h, got = run(wl, topk)
    check_layout(topk.numpy(), wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                 wl.alignment, wl.recv_capacity, got["cnt"], got["tok_per_rank"],
                 got["psum_expert"], got["psum_rank"], got["dst_slot"], got["meta"],
                 got["num_recv"])
    assert h.status() == 0


EDGE = {
    "masked": dict(base="decode", mask_frac=0.2),
    "ragged": dict(base="decode", num_tokens=1000),
    "one_range": dict(base="tiny", num_tokens=77),
    "one_token": dict(base="tiny", num_tokens=1),
    "generic_k5": dict(base="tiny", topk=5, hidden=384, alignment=3),
    "k1": dict(base="tiny", topk=1, alignment=8),
    "k16": dict(base="tiny", topk=16, num_expert_per_rank=16, alignment=16),
    "max_experts": dict(base="tiny", world_size=64, num_expert_per_rank=32, max_tok_per_rank=64,
                        num_tokens=4096, topk=8, alignment=2),
    "epr1": dict(base="tiny", num_expert_per_rank=1, topk=4, alignment=2),
    "epr7": dict(base="tiny", world_size=3, num_expert_per_rank=7, max_tok_per_rank=64,
                 num_tokens=150, alignment=5),
    "zipf_hot": dict(base="skewed", num_tokens=4096),
    # 262080 padding rows: 32 CTAs for 8 ranges of tokens (the others only fill)
    "big_alignment": dict(base="decode", alignment=4096),
    # more experts than one warp scans (600): the block-wide scans, no presort
    "experts_600": dict(base="prefill_bf16", num_expert_per_rank=75, max_tok_per_rank=512,
                        num_tokens=4096, alignment=4),
    # 17 superchunks of 16 ranges and a ragged last range
    "superchunks": dict(base="prefill_bf16", max_tok_per_rank=4352, num_tokens=34800),
}


def edge_wl(spec):
    spec = dict(spec)
    base = synth.WORKLOADS[spec.pop("base")]
    mask = spec.pop("mask_frac", 0.0)
    return base.with_(**spec), mask


# 2048 experts: 16 per-warp histograms of E+W counts need ~200 KB of shared
# memory, beyond the single-launch kernels' limit: the three launches serve
TOO_WIDE = {"max_experts"}


@pytest.mark.parametrize("case", list(EDGE))
def test_fused_layout_edge_cases(case, fused):
    wl, mask = edge_wl(EDGE[case])
    topk = synth.gen_topk(wl, mask_frac=mask)
    h, _ = run(wl, topk, expect="launches" if case in TOO_WIDE else "fused")
    assert h.status() == 0


def test_fused_out_of_range_ids_are_skipped_and_flagged(fused):
    wl = synth.WORKLOADS["skewed"].with_(num_tokens=3000)
    topk = synth.gen_topk(wl)
    topk[3, 1] = wl.num_experts
    topk[2500, 0] = -5
    topk[9, 2] = -1
    h, _ = run(wl, topk)
    assert h.status() == ep.ERR_BAD_EXPERT


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed", "prefill_bf16", "masked", "ragged",
                                  "generic_k5", "epr7", "k16"])
def test_fused_nonexpand_layout(name, fused):
    spec = EDGE.get(name, dict(base=name))
    wl, mask = edge_wl(spec)
    topk = synth.gen_topk(wl, mask_frac=mask)
    h, _ = run(wl, topk, no_expand=True)
    assert h.status() == 0


def test_fused_many_launches_on_one_handle(fused):
    """Launches of changing size in a row on one handle, without
    synchronising in between: each launch's barrier must start from the state
    the previous one left, and each must add into a zeroed superchunk buffer.
    Outputs are compared after each launch."""
    wl = synth.WORKLOADS["prefill_bf16"]
    h = ep.EpHandle(cfg_of(wl))
    sizes = [32768, 2000, 31000, 129, 32768, 4096, 1, 16384, 32768]
    for i, n in enumerate(sizes):
        w = wl.with_(num_tokens=n, seed=wl.seed + i)
        topk = synth.gen_topk(w, mask_frac=0.05 * (i % 2))
        h.layout(topk.cuda())
        assert ran_path(h.variant(0)) == "fused", h.variant(0)
        assert_layout_equal(gpu_fields(h), ref_layout(w, topk.numpy()), n)
    # and several launches queued back to back, only the last one compared
    topks = [synth.gen_topk(wl.with_(num_tokens=n, seed=99 + n)) for n in (5000, 32768, 777, 20000)]
    dev = [t.cuda() for t in topks]
    for t in dev:
        h.layout(t)
    last = wl.with_(num_tokens=20000, seed=99 + 20000)
    assert_layout_equal(gpu_fields(h), ref_layout(last, topks[-1].numpy()), "queued")
    assert h.status() == 0


def test_fused_layout_then_dispatch_and_combine(fused):
    """The fused layout lets the dispatch after it be scheduled early; the
    dispatch waits for the layout's completion before it reads dst_slot."""
    wl = synth.WORKLOADS["skewed"]
    case = synth.make_case(wl, device="cuda")
    h = ep.EpHandle(cfg_of(wl))
    recv = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((wl.num_tokens, wl.hidden), dtype=torch.bfloat16, device="cuda")
    h.layout(case["topk_idx"].cuda())
    h.dispatch(case["x"], recv)
    h.combine(recv, case["topk_weights"].cuda(), out)
    torch.cuda.synchronize()
    assert ran_path(h.variant(0)) == "fused", h.variant(0)
    ref = ref_layout(wl, case["topk_idx"].numpy())
    real = ref["dst_slot"][ref["dst_slot"] >= 0]
    want = np.zeros((wl.recv_capacity, wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], want)
    got = synth.bits16(recv)
    assert np.array_equal(got[real], want[real])
    y = synth.bits16(recv)
    w = case["topk_weights"].cpu().numpy()
    want_out = oracle.combine(y, ref["dst_slot"], w)
    assert np.array_equal(synth.bits16(out), want_out)
    assert h.status() == 0


def test_fused_barrier_wait_limit_gives_up_cleanly(monkeypatch):
    """A wait limit of 0 makes every CTA but the last to arrive give up at the
    grid barrier (the deadline is checked before the generation): those CTAs
    record value 2 (bit 1) in the device error word and return.  Every CTA
    still arrived, so the barrier state stays consistent: the same process then
    builds a handle with the default limit and gets the oracle's layout, and
    the timed-out handle itself keeps launching without hanging."""
    set_layout_path(monkeypatch, "fused")
    wl = synth.WORKLOADS["prefill_bf16"]
    topk = synth.gen_topk(wl)
    monkeypatch.setenv("EP_GB300_WAIT_NS", "0")
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    torch.cuda.synchronize()
    assert ran_path(h.variant(0)) == "fused", h.variant(0)
    assert h.status() == ep.ERR_TIMEOUT
    assert h.status() == 0                      # reading clears it
    h.layout(topk.cuda())
    assert h.status() == ep.ERR_TIMEOUT
    monkeypatch.delenv("EP_GB300_WAIT_NS")
    h2 = ep.EpHandle(cfg_of(wl))
    h2.layout(topk.cuda())
    assert_layout_equal(gpu_fields(h2), ref_layout(wl, topk.numpy()))
    assert h2.status() == 0


def test_fused_layouts_on_two_streams_at_once(fused):
    """Two handles, each on its own stream, launch their cooperative layouts
    back to back without synchronising, so the two grids run at the same time
    where the GPU has room: each keeps its barrier and sums in its own handle,
    and both give the oracle's layout."""
    a = synth.WORKLOADS["prefill_bf16"]
    b = synth.WORKLOADS["skewed"]
    ha, hb = ep.EpHandle(cfg_of(a)), ep.EpHandle(cfg_of(b))
    ta, tb = synth.gen_topk(a), synth.gen_topk(b, mask_frac=0.05)
    da, db = ta.cuda(), tb.cuda()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(20):
        ha.layout(da, stream=sa)
        hb.layout(db, stream=sb)
    torch.cuda.synchronize()
    assert ran_path(ha.variant(0)) == "fused" and ran_path(hb.variant(0)) == "fused"
    assert_layout_equal(gpu_fields(ha), ref_layout(a, ta.numpy()), "a")
    assert_layout_equal(gpu_fields(hb), ref_layout(b, tb.numpy()), "b")
    assert ha.status() == 0 and hb.status() == 0
