"""ep_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (their memory belongs to another framework's pool, or they must
not allocate after start-up).  It takes every output from the caller and keeps
its scratch in a fixed array inside the library.

Checked against the handle-based ep_layout, which allocates its scratch with
cudaMalloc: the outputs must be the same bytes, on two calls in a row with
different routings (the shared scratch keeps the previous call's contents).
This file is collected last, and passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth


@pytest.fixture(scope="module")
def gpu():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def cfg_of(wl):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, wl.dispatch_dtype, wl.use_weights)


def noalloc_outputs(wl, n):
    dev = "cuda"
    E, W, K = wl.num_experts, wl.world_size, wl.topk
    shapes = {"num_unaligned_per_expert": (E,), "num_tokens_per_rank": (W,),
              "psum_per_expert": (E + 1,), "psum_per_rank": (W + 1,), "num_recv": (1,),
              "dst_slot": (max(n, 1), K), "recv_src_metadata": (wl.recv_capacity, K + 2),
              "device_error": (1,)}
    # filled with a pattern so that an output the call fails to write shows up
    return {k: torch.full(s, -12345, dtype=torch.int32, device=dev) for k, s in shapes.items()}


PAIRS = [
    ("num_unaligned_per_expert", ep.FIELD_NUM_UNALIGNED_PER_EXPERT),
    ("num_tokens_per_rank", ep.FIELD_NUM_TOKENS_PER_RANK),
    ("psum_per_expert", ep.FIELD_PSUM_PER_EXPERT),
    ("psum_per_rank", ep.FIELD_PSUM_PER_RANK),
    ("num_recv", ep.FIELD_NUM_RECV),
    ("dst_slot", ep.FIELD_DST_SLOT),
    ("recv_src_metadata", ep.FIELD_RECV_SRC_METADATA),
]


@pytest.mark.gpu
def test_noalloc_layout_matches_the_allocating_layout_on_two_calls_in_a_row(gpu):
    # small batches run the single-launch cluster kernel, large ones the three
    # launches that use the static scratch
    calls = [synth.WORKLOADS["decode"], synth.WORKLOADS["prefill_bf16"], synth.WORKLOADS["skewed"],
             synth.WORKLOADS["decode"].with_(num_tokens=1000, alignment=16)]
    for wl in calls:                       # one call after another on the same static scratch
        topk = synth.gen_topk(wl, mask_frac=0.01).cuda()
        out = noalloc_outputs(wl, wl.num_tokens)
        ep.ep_layout_noalloc(cfg_of(wl), topk, out)
        h = ep.EpHandle(cfg_of(wl))
        h.layout(topk)
        torch.cuda.synchronize()
        assert_same_as_handle(out, h, wl)
        h.free()


def assert_same_as_handle(out, h, wl):
    """The no-alloc outputs equal the allocating handle's fields, bit for bit."""
    n = wl.num_tokens
    for name, field in PAIRS:
        want = h.field(field).cpu().numpy()
        got = out[name].cpu().numpy()
        if name == "dst_slot":
            got = got[:n]
        assert np.array_equal(got, want), (wl.name, name)   # integer outputs: bit-exact
    assert int(out["device_error"].cpu()[0]) == 0
    assert h.status() == 0


@pytest.mark.gpu
def test_noalloc_empty_batch_and_small_large_small(gpu):
    """N = 0 (count skipped: the other kernels still write zero counts and -1
    metadata), then a batch that takes the cluster kernel, one that uses the
    static scratch, and a small one again, each against the allocating layout."""
    dec = synth.WORKLOADS["decode"].with_(alignment=16)
    calls = [dec.with_(num_tokens=0), dec.with_(num_tokens=700),
             synth.WORKLOADS["prefill_bf16"], dec.with_(num_tokens=0),
             synth.WORKLOADS["skewed"], dec.with_(num_tokens=33)]
    for i, wl in enumerate(calls):
        topk = synth.gen_topk(wl.with_(seed=wl.seed + i), mask_frac=0.02).cuda()
        out = noalloc_outputs(wl, wl.num_tokens)
        ep.ep_layout_noalloc(cfg_of(wl), topk, out)
        h = ep.EpHandle(cfg_of(wl))
        h.layout(topk)
        torch.cuda.synchronize()
        assert_same_as_handle(out, h, wl)
        if wl.num_tokens == 0:
            assert int(out["num_recv"].cpu()[0]) == 0
            assert bool((out["recv_src_metadata"] == -1).all())
        h.free()


@pytest.mark.gpu
def test_noalloc_at_the_scratch_limit_matches_the_oracle(gpu):
    """The largest batch the static scratch admits for 256 experts over 8 ranks:
    3*(E+W)*ceil(N/128) + (E+W) <= 262144 gives ceil(N/128) <= 330, N = 42240.
    Compared with the CPU oracle directly; one token more is rejected."""
    wl = synth.WORKLOADS["prefill_bf16"].with_(max_tok_per_rank=5288, num_tokens=42240)
    E, W = wl.num_experts, wl.world_size
    assert 3 * (E + W) * 330 + (E + W) <= 262144 < 3 * (E + W) * 331 + (E + W)
    topk = synth.gen_topk(wl, mask_frac=0.01)
    out = noalloc_outputs(wl, wl.num_tokens)
    ep.ep_layout_noalloc(cfg_of(wl), topk.cuda(), out)
    torch.cuda.synchronize()
    ref = oracle.layout(topk.numpy(), W, wl.max_tok_per_rank, wl.num_expert_per_rank,
                        wl.alignment)
    want = {"num_unaligned_per_expert": ref["cnt"], "num_tokens_per_rank": ref["tok_per_rank"],
            "psum_per_expert": ref["psum_expert"], "psum_per_rank": ref["psum_rank"],
            "num_recv": np.array([ref["num_recv"]]), "dst_slot": ref["dst_slot"],
            "recv_src_metadata": ref["meta"]}
    for k, v in want.items():
        assert np.array_equal(out[k].cpu().numpy(), np.asarray(v)), k
    assert int(out["device_error"].cpu()[0]) == 0
    # one token past the limit: 331 chunks
    over = wl.with_(num_tokens=42241)
    big = noalloc_outputs(over, over.num_tokens)
    with pytest.raises(ep.EpError) as e:
        ep.ep_layout_noalloc(cfg_of(over), synth.gen_topk(over).cuda(), big)
    assert e.value.code == ep.EP_EINVAL and "static scratch" in str(e.value)


@pytest.mark.gpu
def test_noalloc_reports_bad_expert_ids(gpu):
    wl = synth.WORKLOADS["tiny"]
    topk = synth.gen_topk(wl)
    topk[0, 0] = wl.num_experts + 3
    out = noalloc_outputs(wl, wl.num_tokens)
    ep.ep_layout_noalloc(cfg_of(wl), topk.cuda(), out)
    torch.cuda.synchronize()
    assert int(out["device_error"].cpu()[0]) == ep.ERR_BAD_EXPERT
    assert int(out["dst_slot"].cpu()[0, 0]) == -1


def test_noalloc_rejects_requests_beyond_the_static_scratch():
    # 64 ranks x 32 experts and 16384 tokens: 3*(2048+64)*128 + 2112 int32 > 262144
    cfg = ep.make_cfg(64, 1024, 256, 32, 8, 1, "bf16", True)
    L = ep.load_library()
    dummy = ctypes.c_void_p(256)          # never dereferenced: the size check comes first
    rc = L.ep_layout_noalloc(ctypes.byref(cfg), dummy, 16384, *([dummy] * 8), None)
    assert rc == ep.EP_EINVAL
    assert "static scratch" in ep.ep_last_error()
