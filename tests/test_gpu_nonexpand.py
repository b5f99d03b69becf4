"""GPU parity of the non-expand layout (EPHandle do_expand = false: one receive
row per (token, destination rank)) and of dispatch / forwarding / combine over
its rows, through the C ABI, against the CPU oracle.  All bit-exact."""
import numpy as np
import pytest
import torch

import combine_ep_layout_gb300 as ep
import oracle
import synth
from layout_checks import check_layout_nonexpand, LAYOUT_PATHS, set_layout_path, ran_path

pytestmark = pytest.mark.gpu

FIELDS = {
    "cnt": ep.FIELD_NUM_UNALIGNED_PER_EXPERT,
    "tok_per_rank": ep.FIELD_NUM_TOKENS_PER_RANK,
    "psum_expert": ep.FIELD_PSUM_PER_EXPERT,
    "psum_rank": ep.FIELD_PSUM_PER_RANK,
    "dst_slot": ep.FIELD_DST_SLOT,
    "send_slot": ep.FIELD_SEND_SLOT,
    "meta": ep.FIELD_RECV_SRC_METADATA,
}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def cfg_of(wl, dtype="bf16"):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, dtype, False, no_expand=True)


def ref_layout(wl, topk):
    return oracle.layout_nonexpand(np.asarray(topk), wl.world_size, wl.max_tok_per_rank,
                                   wl.num_expert_per_rank, wl.alignment)


def gpu_fields(h):
    torch.cuda.synchronize()
    out = {k: h.field(f).cpu().numpy() for k, f in FIELDS.items()}
    out["num_recv"] = int(h.field(ep.FIELD_NUM_RECV).cpu()[0])
    return out


def assert_equal(got, ref):
    for k in list(FIELDS) + ["num_recv"]:
        assert np.array_equal(np.asarray(got[k]), np.asarray(ref[k])), k


EDGE = {
    "tiny": dict(base="tiny"),
    "decode": dict(base="decode"),
    "skewed": dict(base="skewed"),
    "prefill": dict(base="prefill_bf16"),
    "masked": dict(base="decode", mask_frac=0.3),
    "ragged": dict(base="decode", num_tokens=1000),
    "one_token": dict(base="tiny", num_tokens=1),
    "no_tokens": dict(base="tiny", num_tokens=0),
    "k_above_w": dict(base="tiny", world_size=2, num_expert_per_rank=16, topk=8,
                      max_tok_per_rank=64),
    "w1": dict(base="tiny", world_size=1, num_expert_per_rank=32, max_tok_per_rank=128),
    "generic_k5": dict(base="tiny", topk=5, hidden=384, alignment=3),
    "k16_w64": dict(base="tiny", world_size=64, num_expert_per_rank=32, max_tok_per_rank=64,
                    num_tokens=4096, topk=16, alignment=2),
    "epr1": dict(base="tiny", num_expert_per_rank=1, topk=4),
    "epr7": dict(base="tiny", world_size=3, num_expert_per_rank=7, max_tok_per_rank=64,
                 num_tokens=150),
}


def edge_wl(spec):
    spec = dict(spec)
    base = synth.WORKLOADS[spec.pop("base")]
    mask = spec.pop("mask_frac", 0.0)
    return (base.with_(**spec) if spec else base), mask


@pytest.mark.parametrize("case", list(EDGE))
def test_layout_bit_exact(case):
    wl, mask = edge_wl(EDGE[case])
    topk = synth.gen_topk(wl, mask_frac=mask)
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    got = gpu_fields(h)
    ref = ref_layout(wl, topk.numpy())
    assert got["meta"].shape[0] == ref["rcap"] == ep.ep_recv_capacity(cfg_of(wl))
    assert_equal(got, ref)
    if wl.num_tokens <= 4096:
        check_layout_nonexpand(topk.numpy(), wl.world_size, wl.max_tok_per_rank,
                               wl.num_expert_per_rank, wl.alignment, ref["rcap"], got["cnt"],
                               got["tok_per_rank"], got["psum_expert"], got["psum_rank"],
                               got["dst_slot"], got["send_slot"], got["meta"], got["num_recv"])
    assert h.status() == 0
    assert h.variant(0).startswith("ep_layout_nonexpand_")


def test_duplicates_and_bad_ids():
    wl = synth.WORKLOADS["tiny"]
    g = torch.Generator().manual_seed(5)
    topk = torch.randint(-1, wl.num_experts, (wl.num_tokens, wl.topk), generator=g)
    topk[3, 0] = wl.num_experts + 2
    topk[7, :] = topk[7, 0]
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    assert_equal(gpu_fields(h), ref_layout(wl, topk.numpy()))
    assert h.status() == ep.ERR_BAD_EXPERT


@pytest.mark.parametrize("name,dtype", [("tiny", "bf16"), ("decode", "fp8"), ("skewed", "bf16"),
                                        ("decode", "fp4x2"), ("tiny", "fp32")])
def test_dispatch_and_forwarding(name, dtype):
    wl = synth.WORKLOADS[name]
    case = synth.make_case(wl, device="cuda", mask_frac=0.05)
    topk, w = case["topk_idx"], case["topk_weights"]
    cfg = cfg_of(wl, dtype)
    h = ep.EpHandle(cfg)
    h.layout(topk.cuda())
    ref = ref_layout(wl, topk.numpy())
    R, H, K = ref["rcap"], wl.hidden, wl.topk
    rw = torch.full((R, K), -3.0, device="cuda")
    ri = torch.full((R, K), -9, dtype=torch.int32, device="cuda")
    if dtype == "fp8":
        recv = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
        scales = torch.full((R, H // 128), -1.0, dtype=torch.float32, device="cuda")
        h.dispatch(case["x"], recv, scales, w.cuda(), rw, ri)
        torch.cuda.synchronize()
        rq = np.zeros((R, H), np.uint8)
        rs = np.full((R, H // 128), -1.0, np.float32)
        oracle.dispatch_fp8(synth.bits16(case["x"]), ref["send_slot"], rq, rs)
        assert np.array_equal(recv.cpu().numpy(), rq)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    elif dtype == "bf16":
        recv = torch.full((R, H), -7.0, dtype=torch.bfloat16, device="cuda")
        h.dispatch(case["x"], recv, None, w.cuda(), rw, ri)
        torch.cuda.synchronize()
        rx = np.full((R, H), synth.bits16(torch.tensor([-7.0], dtype=torch.bfloat16))[0], np.uint16)
        oracle.dispatch_bf16(synth.bits16(case["x"]), ref["send_slot"], rx)
        assert np.array_equal(synth.bits16(recv), rx)
    else:
        rb = 4 * H if dtype == "fp32" else H // 2
        x = torch.randint(0, 256, (wl.num_tokens, rb), dtype=torch.uint8, device="cuda",
                          generator=torch.Generator(device="cuda").manual_seed(3))
        recv = torch.full((R, rb), 0x5A, dtype=torch.uint8, device="cuda")
        xin = x.view(torch.float32) if dtype == "fp32" else x
        h.dispatch(xin, recv, None, w.cuda(), rw, ri)
        torch.cuda.synchronize()
        want = np.full((R, rb), 0x5A, np.uint8)
        oracle.dispatch_bytes(x.cpu().numpy(), ref["send_slot"], want)
        assert np.array_equal(recv.cpu().numpy(), want)
    want_w = np.full((R, K), -3.0, np.float32)
    want_i = np.full((R, K), -9, np.int32)
    oracle.forward_routing_nonexpand(topk.numpy(), w.numpy(), ref["dst_slot"], ref["send_slot"],
                                     want_w, want_i)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), want_w.view(np.uint32))
    assert np.array_equal(ri.cpu().numpy(), want_i)
    assert h.status() == 0


@pytest.mark.parametrize("name,use_bias,out_dtype", [("tiny", False, "bf16"), ("tiny", True, "fp32"),
                                                     ("decode", True, "bf16"),
                                                     ("skewed", False, "fp32")])
def test_combine(name, use_bias, out_dtype):
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl, mask_frac=0.05)
    ref = ref_layout(wl, topk.numpy())
    R = ref["rcap"]
    valid = np.zeros(R, bool)
    valid[:ref["num_recv"]] = True
    y = synth.gen_bf16_normal(R, wl.hidden, seed=wl.seed * 16 + 3, device="cuda")
    y[torch.from_numpy(~valid).cuda()] = float("nan")      # rows nobody sends must not be read
    bias = synth.gen_bf16_normal(wl.num_tokens, wl.hidden, seed=wl.seed * 16 + 7, device="cuda")
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    dt = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    out = torch.full((wl.num_tokens, wl.hidden), -1, dtype=dt, device="cuda")
    h.combine(y, None, out, bias if use_bias else None)
    torch.cuda.synchronize()
    want = oracle.combine_ex(synth.bits16(y), ref["send_slot"], None,
                             synth.bits16(bias) if use_bias else None, out_dtype)
    if out_dtype == "fp32":
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bits16(out), want)


def test_identity_round_trip_prefill():
    # dispatch then combine the received rows unchanged: bf16(n_t * x[t]) where
    # n_t is the number of ranks token t reached (exact in fp32 for n_t <= 8)
    wl = synth.WORKLOADS["prefill_bf16"]
    case = synth.make_case(wl, device="cuda")
    h = ep.EpHandle(cfg_of(wl))
    h.layout(case["topk_idx"].cuda())
    R = ep.ep_recv_capacity(cfg_of(wl))
    recv = torch.empty((R, wl.hidden), dtype=torch.bfloat16, device="cuda")
    h.dispatch(case["x"], recv)
    out = torch.empty_like(case["x"])
    h.combine(recv, None, out)
    n = (h.field(ep.FIELD_SEND_SLOT) >= 0).sum(dim=1, keepdim=True).float()
    want = (case["x"].float() * n).to(torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("path", LAYOUT_PATHS)
@pytest.mark.parametrize("case", ["tiny", "masked", "ragged", "one_token", "k_above_w", "w1",
                                  "generic_k5", "epr7", "full_2048"])
def test_small_batch_layout_both_paths(case, path, monkeypatch):
    set_layout_path(monkeypatch, path)
    spec = EDGE.get(case, dict(base="decode", max_tok_per_rank=256, num_tokens=2048))
    wl, mask = edge_wl(spec)
    topk = synth.gen_topk(wl, mask_frac=mask)
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    assert_equal(gpu_fields(h), ref_layout(wl, topk.numpy()))
    assert ran_path(h.variant(0)) == path, h.variant(0)
    assert h.status() == 0
