"""The TMA-staged dispatch (EP_GB300_DISPATCH_TMA=1): rows brought into shared
memory by bulk copies and written to their receive rows by bulk copies, for
the byte-copy transports.  The same bytes as the oracle's dispatch, with the
same layouts and forwarding as the register copy; and its bounded mbarrier
waits give up cleanly (device error value 2) when the wait limit is 0."""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.fixture
def tma(monkeypatch):
    monkeypatch.setenv("EP_GB300_DISPATCH_TMA", "1")   # read when a handle is built


def cfg_of(wl, dtype="bf16", no_expand=False):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, dtype, wl.use_weights and not no_expand,
                       no_expand=no_expand)


def ref_layout(wl, topk):
    return oracle.layout(np.asarray(topk), wl.world_size, wl.max_tok_per_rank,
                         wl.num_expert_per_rank, wl.alignment)


CASES = {
    "tiny": dict(base="tiny"),
    "decode_masked": dict(base="decode", mask=0.1),
    "ragged": dict(base="decode", num_tokens=1000),
    "prefill_4096": dict(base="prefill_bf16", num_tokens=4096, max_tok_per_rank=512),
    "skewed_2048": dict(base="skewed", num_tokens=2048, max_tok_per_rank=256),
    "generic_k5": dict(base="tiny", topk=5, hidden=384, alignment=3),
    "one_token": dict(base="tiny", num_tokens=1),
}


def case_wl(name):
    spec = dict(CASES[name])
    base = synth.WORKLOADS[spec.pop("base")]
    mask = spec.pop("mask", 0.0)
    return base.with_(**spec), mask


@pytest.mark.parametrize("name", list(CASES))
def test_tma_dispatch_bf16_matches_the_oracle(name, tma):
    wl, mask = case_wl(name)
    case = synth.make_case(wl, device="cuda", mask_frac=mask)
    h = ep.EpHandle(cfg_of(wl))
    assert h.variant(1) == "ep_dispatch_tma_bf16"
    h.layout(case["topk_idx"].cuda())
    recv = torch.full((wl.recv_capacity, wl.hidden), -1, dtype=torch.int16,
                      device="cuda").view(torch.bfloat16)
    h.dispatch(case["x"], recv)
    torch.cuda.synchronize()
    ref = ref_layout(wl, case["topk_idx"].numpy())
    want = np.full((wl.recv_capacity, wl.hidden), 0xFFFF, np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], want)
    assert np.array_equal(synth.bits16(recv), want)
    assert h.status() == 0


@pytest.mark.parametrize("dtype", ["fp32", "fp4x2"])
def test_tma_dispatch_opaque_transports(dtype, tma):
    wl = synth.WORKLOADS["decode"]
    topk = synth.gen_topk(wl, mask_frac=0.05)
    row_bytes = 4 * wl.hidden if dtype == "fp32" else wl.hidden // 2
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randint(0, 256, (wl.num_tokens, row_bytes), dtype=torch.uint8, device="cuda", generator=g)
    h = ep.EpHandle(cfg_of(wl, dtype))
    assert h.variant(1) == "ep_dispatch_tma_" + dtype
    h.layout(topk.cuda())
    recv = torch.full((wl.recv_capacity, row_bytes), 0x5A, dtype=torch.uint8, device="cuda")
    h.dispatch(x.view(torch.float32) if dtype == "fp32" else x, recv)
    torch.cuda.synchronize()
    want = np.full((wl.recv_capacity, row_bytes), 0x5A, np.uint8)
    oracle.dispatch_bytes(x.cpu().numpy(), ref_layout(wl, topk.numpy())["dst_slot"], want)
    assert np.array_equal(recv.cpu().numpy(), want)
    assert h.status() == 0


def test_tma_dispatch_forwarding_and_nonexpand(tma):
    wl = synth.WORKLOADS["decode"].with_(use_weights=False)
    case = synth.make_case(wl, device="cuda", mask_frac=0.05)
    topk, w = case["topk_idx"], case["topk_weights"]
    # expand layout with forwarded routing
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    R = wl.recv_capacity
    recv = torch.zeros((R, wl.hidden), dtype=torch.bfloat16, device="cuda")
    rw = torch.full((R,), -3.0, dtype=torch.float32, device="cuda")
    ri = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    h.dispatch(case["x"], recv, topk_weights=w.cuda(), recv_topk_weights=rw, recv_topk_idx=ri)
    torch.cuda.synchronize()
    ref = ref_layout(wl, topk.numpy())
    ww = np.full(R, -3.0, np.float32)
    wi = np.full(R, -7, np.int32)
    oracle.forward_routing(topk.numpy(), w.numpy(), ref["dst_slot"], ww, wi)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ww.view(np.uint32))
    assert np.array_equal(ri.cpu().numpy(), wi)
    # non-expand layout: one row per (token, destination rank)
    hn = ep.EpHandle(cfg_of(wl, no_expand=True))
    assert hn.variant(1) == "ep_dispatch_tma_bf16"
    hn.layout(topk.cuda())
    Rn = ep.ep_recv_capacity(cfg_of(wl, no_expand=True))
    rn = torch.full((Rn, wl.hidden), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    hn.dispatch(case["x"], rn)
    torch.cuda.synchronize()
    refn = oracle.layout_nonexpand(topk.numpy(), wl.world_size, wl.max_tok_per_rank,
                                   wl.num_expert_per_rank, wl.alignment)
    want = np.full((Rn, wl.hidden), 0xFFFF, np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), refn["send_slot"], want)
    assert np.array_equal(synth.bits16(rn), want)
    assert h.status() == 0 and hn.status() == 0


def test_rows_too_large_for_two_stages_take_the_register_copy(tma):
    # fp32 rows of 32768 channels (128 KB): two ring stages do not fit in shared memory
    wl = synth.WORKLOADS["tiny"].with_(hidden=32768, num_tokens=8)
    h = ep.EpHandle(cfg_of(wl, "fp32"))
    assert not h.variant(1).startswith("ep_dispatch_tma")


def test_tma_wait_limit_gives_up_cleanly(monkeypatch, tma):
    """A wait limit of 0 makes every CTA give up at its first mbarrier test (the
    first row is still being copied): the kernel records value 2 (bit 1) in the
    device error word, waits for its own copies and returns; the context stays
    usable and a handle with the default limit then dispatches correctly."""
    wl = synth.WORKLOADS["decode"]
    case = synth.make_case(wl, device="cuda")
    monkeypatch.setenv("EP_GB300_WAIT_NS", "0")
    h = ep.EpHandle(cfg_of(wl))
    h.layout(case["topk_idx"].cuda())
    recv = torch.zeros((wl.recv_capacity, wl.hidden), dtype=torch.bfloat16, device="cuda")
    h.dispatch(case["x"], recv)
    assert h.status() == ep.ERR_TIMEOUT
    assert h.status() == 0                      # reading clears it
    monkeypatch.delenv("EP_GB300_WAIT_NS")
    h2 = ep.EpHandle(cfg_of(wl))
    h2.layout(case["topk_idx"].cuda())
    h2.dispatch(case["x"], recv)
    torch.cuda.synchronize()
    ref = ref_layout(wl, case["topk_idx"].numpy())
    want = np.zeros((wl.recv_capacity, wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], want)
    assert np.array_equal(synth.bits16(recv), want)
    assert h2.status() == 0
