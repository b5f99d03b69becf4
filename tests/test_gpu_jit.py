"""GPU parity of the run-time specialisations: a shape outside the compiled
table (hidden 2560, top-5) runs NVRTC-compiled kernels, bit-exact against the
oracle, and the same bytes as the compiled generic variant."""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["tiny"].with_(world_size=4, max_tok_per_rank=64, num_tokens=250,
                                   hidden=2560, num_expert_per_rank=8, topk=5, alignment=2)


@pytest.fixture(scope="module", autouse=True)
def built(tmp_path_factory):
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.fixture()
def cache(tmp_path, monkeypatch):
    monkeypatch.setenv("EP_GB300_JIT_CACHE", str(tmp_path / "jit"))


def cfg(dtype, use_w=True):
    return ep.make_cfg(WL.world_size, WL.hidden, WL.max_tok_per_rank, WL.num_expert_per_rank,
                       WL.topk, WL.alignment, dtype, use_w)


def run(dtype, use_w=True):
    case = synth.make_case(WL, device="cuda", mask_frac=0.05)
    h = ep.EpHandle(cfg(dtype, use_w))
    h.layout(case["topk_idx"].cuda())
    R, H = WL.recv_capacity, WL.hidden
    if dtype == "fp8":
        recv = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
        sc = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
    else:
        recv = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
        sc = None
    h.dispatch(case["x"], recv, sc)
    y = synth.gen_bf16_normal(R, H, seed=17, device="cuda")
    out = torch.zeros_like(case["x"])
    h.combine(y, case["topk_weights"].cuda() if use_w else None, out)
    torch.cuda.synchronize()
    assert h.status() == 0
    return h, case, recv, sc, y, out


def test_jit_kernels_match_the_oracle(cache):
    h, case, recv, _, y, out = run("bf16")
    if not h.variant(1).startswith("ep_jit_"):
        pytest.skip("run-time specialisation unavailable: " + h.variant(1))
    assert h.variant(1) == "ep_jit_dispatch_copy_rb5120_k5"
    assert h.variant(2) == "ep_jit_combine_w_h2560_k5"
    ref = oracle.layout(case["topk_idx"].numpy(), WL.world_size, WL.max_tok_per_rank,
                        WL.num_expert_per_rank, WL.alignment)
    rx = np.zeros((WL.recv_capacity, WL.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], rx)
    assert np.array_equal(synth.bits16(recv), rx)
    want = oracle.combine(synth.bits16(y), ref["dst_slot"], case["topk_weights"].numpy())
    assert np.array_equal(synth.bits16(out), want)


def test_jit_fp8_and_unweighted_combine(cache):
    h, case, recv, sc, y, out = run("fp8", use_w=False)
    if not h.variant(1).startswith("ep_jit_"):
        pytest.skip("run-time specialisation unavailable")
    assert h.variant(1) == "ep_jit_dispatch_fp8_h2560_k5"
    assert h.variant(2) == "ep_jit_combine_h2560_k5"
    ref = oracle.layout(case["topk_idx"].numpy(), WL.world_size, WL.max_tok_per_rank,
                        WL.num_expert_per_rank, WL.alignment)
    q = np.zeros((WL.recv_capacity, WL.hidden), np.uint8)
    s = np.zeros((WL.recv_capacity, WL.hidden // 128), np.float32)
    oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], q, s)
    assert np.array_equal(recv.cpu().numpy(), q)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert np.array_equal(synth.bits16(out), oracle.combine(synth.bits16(y), ref["dst_slot"], None))


def test_generic_variant_gives_the_same_bytes(cache, monkeypatch):
    h1, c1, r1, _, y1, o1 = run("bf16")
    monkeypatch.setenv("EP_GB300_JIT", "0")
    h2, c2, r2, _, y2, o2 = run("bf16")
    assert h2.variant(1) == "ep_dispatch_bf16_generic" and h2.variant(2) == "ep_combine_w_generic"
    assert torch.equal(r1.view(torch.int16), r2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_jit_kernels_replay_in_a_cuda_graph(cache):
    h = ep.EpHandle(cfg("bf16"))
    if not h.variant(1).startswith("ep_jit_"):
        pytest.skip("run-time specialisation unavailable")
    case = synth.make_case(WL, device="cuda")
    topk = case["topk_idx"].cuda()
    recv = torch.zeros((WL.recv_capacity, WL.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(case["x"])
    w = case["topk_weights"].cuda()
    h.layout(topk)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h.layout(topk, stream=s)
        h.dispatch(case["x"], recv, stream=s)
        h.combine(recv, w, out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.layout(case["topk_idx"].numpy(), WL.world_size, WL.max_tok_per_rank,
                        WL.num_expert_per_rank, WL.alignment)
    rx = np.zeros((WL.recv_capacity, WL.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], rx)
    assert np.array_equal(synth.bits16(out), oracle.combine(rx, ref["dst_slot"], case["topk_weights"].numpy()))
