"""The TMA combine (EP_GB300_COMBINE_TMA=1: each token's K expert rows staged in
shared memory by bulk copies, piece by piece) against the CPU oracle, bit for
bit: the same fixed fma order as the register combine.  Cases: every workload
shape with and without weights, masked entries, the non-expand layout, the
top-k edge cases (1, 5, 16) and the whole 32768-token prefill batch.  A wait
limit of 0 makes the copies' wait give up: the kernel reports device error
value 2 (bit 1), stores nothing and leaves the context usable."""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth
from test_gpu_parity import (EDGE, assert_combine_close, combine_case, compact_slots, edge_wl,
                             token_ranges)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tma_combine(monkeypatch):
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    monkeypatch.setenv("EP_GB300_COMBINE_TMA", "1")


def check_served_by_tma(h):
    assert h.variant(2).startswith("ep_combine_tma"), h.variant(2)


@pytest.mark.parametrize("name,use_w,mask", [("tiny", True, 0.0), ("tiny", False, 0.2),
                                             ("decode", True, 0.0), ("decode", False, 0.0),
                                             ("skewed", True, 0.05)])
def test_tma_combine_whole(name, use_w, mask):
    wl = synth.WORKLOADS[name]
    h, ref, y, w, out = combine_case(wl, use_w, mask)
    check_served_by_tma(h)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], w.numpy() if use_w else None)
    assert_combine_close(synth.bits16(out), want)
    assert h.status() == 0


@pytest.mark.parametrize("case_name", ["generic_k5", "k16", "k1", "ragged"])
def test_tma_combine_edge(case_name):
    wl, mask = edge_wl(EDGE[case_name])
    h, ref, y, w, out = combine_case(wl, True, mask)
    check_served_by_tma(h)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], w.numpy())
    assert_combine_close(synth.bits16(out), want)


def test_tma_combine_prefill_whole():
    """Every token of the 32768-token prefill combine (rows cut into 8 pieces of
    1792 bytes) against the oracle, range by range."""
    wl = synth.WORKLOADS["prefill_bf16"]
    h, ref, y, w, out = combine_case(wl)
    check_served_by_tma(h)
    wn = w.numpy()
    for a, b in token_ranges(wl.num_tokens):
        ds = ref["dst_slot"][a:b]
        rows = torch.from_numpy(ds.reshape(-1).astype(np.int64)).cuda()
        want = oracle.combine(synth.bits16(y[rows]), compact_slots(ds), wn[a:b])
        assert_combine_close(synth.bits16(out[a:b]), want)
    assert bool(torch.isfinite(out.float()).all())   # no padding (NaN) row was read


def test_tma_combine_bias_and_fp32_use_the_register_kernel():
    """The TMA combine serves bf16 output without bias; combine_ex with a bias or
    fp32 output still runs (on the register kernel) and matches the oracle."""
    wl = synth.WORKLOADS["decode"]
    topk = synth.gen_topk(wl)
    ref = oracle.layout(topk.numpy(), wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                        wl.alignment)
    y = synth.gen_y(wl, valid_rows=ref["meta"][:, 0] >= 0, device="cuda")
    w = synth.gen_weights(wl)
    h = ep.EpHandle(ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank,
                                wl.num_expert_per_rank, wl.topk, wl.alignment, "bf16", True))
    h.layout(topk.cuda())
    out32 = torch.empty((wl.num_tokens, wl.hidden), dtype=torch.float32, device="cuda")
    h.combine(y, w.cuda(), out32)
    bias = synth.gen_x(wl, device="cuda")
    outb = torch.empty((wl.num_tokens, wl.hidden), dtype=torch.bfloat16, device="cuda")
    h.combine(y, w.cuda(), outb, bias=bias)
    torch.cuda.synchronize()
    want32 = oracle.combine_ex(synth.bits16(y), ref["dst_slot"], w.numpy(), None, "fp32")
    assert np.array_equal(out32.cpu().numpy().view(np.uint32), np.asarray(want32).view(np.uint32))
    wantb = oracle.combine_ex(synth.bits16(y), ref["dst_slot"], w.numpy(), synth.bits16(bias), "bf16")
    assert np.array_equal(synth.bits16(outb), wantb)
    assert h.status() == 0


def test_tma_combine_wait_limit_gives_up_cleanly(monkeypatch):
    """A wait limit of 0: the CTAs give up on their copies at the first test,
    record value 2 (bit 1), let the copies land and return without storing; a
    handle built with the default limit then matches the oracle."""
    wl = synth.WORKLOADS["decode"]
    monkeypatch.setenv("EP_GB300_WAIT_NS", "0")
    h, ref, y, w, out = combine_case(wl)
    check_served_by_tma(h)
    assert h.status() == ep.ERR_TIMEOUT
    assert h.status() == 0
    monkeypatch.delenv("EP_GB300_WAIT_NS")
    h2, ref2, y2, w2, out2 = combine_case(wl)
    want = oracle.combine(synth.bits16(y2), ref2["dst_slot"], w2.numpy())
    assert_combine_close(synth.bits16(out2), want)
    assert h2.status() == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_tma_combine_nonexpand(name):
    """The non-expand layout (one row per (token, destination rank), unweighted):
    the token's rows in ascending rank order, 5% of the entries masked."""
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl, mask_frac=0.05)
    ref = oracle.layout_nonexpand(topk.numpy(), wl.world_size, wl.max_tok_per_rank,
                                  wl.num_expert_per_rank, wl.alignment)
    R = ref["rcap"]
    valid = np.zeros(R, bool)
    valid[:ref["num_recv"]] = True
    y = synth.gen_bf16_normal(R, wl.hidden, seed=wl.seed * 16 + 3, device="cuda")
    y[torch.from_numpy(~valid).cuda()] = float("nan")      # rows nobody sends must not be read
    h = ep.EpHandle(ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank,
                                wl.num_expert_per_rank, wl.topk, wl.alignment, "bf16", False,
                                no_expand=True))
    h.layout(topk.cuda())
    out = torch.full((wl.num_tokens, wl.hidden), -1, dtype=torch.bfloat16, device="cuda")
    h.combine(y, None, out)
    torch.cuda.synchronize()
    check_served_by_tma(h)
    want = oracle.combine_ex(synth.bits16(y), ref["send_slot"], None, None, "bf16")
    assert np.array_equal(synth.bits16(out), want)
    assert h.status() == 0


@pytest.mark.parametrize("kernel", ["register", "tma"])
def test_combine_tokens_with_every_entry_masked(monkeypatch, kernel):
    """Tokens whose K entries are all -1 fold nothing: their output is bf16 +0
    (the fold starts at +0.0f), on both combine kernels; a partly masked token
    folds only its routed rows."""
    monkeypatch.setenv("EP_GB300_COMBINE_TMA", "1" if kernel == "tma" else "0")
    wl = synth.WORKLOADS["decode"]
    topk = synth.gen_topk(wl)
    for t in (0, 5, 17, wl.num_tokens - 1):
        topk[t] = -1
    topk[3, ::2] = -1
    ref = oracle.layout(topk.numpy(), wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                        wl.alignment)
    y = synth.gen_y(wl, valid_rows=ref["meta"][:, 0] >= 0, device="cuda")
    w = synth.gen_weights(wl)
    h = ep.EpHandle(ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank,
                                wl.num_expert_per_rank, wl.topk, wl.alignment, "bf16", True))
    h.layout(topk.cuda())
    out = torch.full((wl.num_tokens, wl.hidden), -1, dtype=torch.bfloat16, device="cuda")
    h.combine(y, w.cuda(), out)
    torch.cuda.synchronize()
    assert h.variant(2).startswith("ep_combine_tma") == (kernel == "tma"), h.variant(2)
    got = synth.bits16(out)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], w.numpy())
    assert np.array_equal(got, want)
    for t in (0, 5, 17, wl.num_tokens - 1):
        assert not got[t].any()
    assert h.status() == 0
