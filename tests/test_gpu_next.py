"""GPU parity of the wider calls against the CPU oracle: routing forwarded with
the rows (ep_dispatch_fwd), the handle's copy of the ids, combine with a bias
and an fp32 output (ep_combine_ex), and the fp32 / packed-fp4 transports.
All bit-exact."""
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


def cfg_of(wl, dtype="bf16", use_weights=True):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, dtype, use_weights)


def ref_layout(wl, topk):
    return oracle.layout(np.asarray(topk), wl.world_size, wl.max_tok_per_rank,
                         wl.num_expert_per_rank, wl.alignment)


@pytest.mark.parametrize("name,dtype,mask", [("tiny", "bf16", 0.2), ("decode", "fp8", 0.0),
                                             ("skewed", "bf16", 0.05)])
def test_dispatch_forwards_the_routing(name, dtype, mask):
    wl = synth.WORKLOADS[name]
    case = synth.make_case(wl, device="cuda", mask_frac=mask)
    topk, w = case["topk_idx"], case["topk_weights"]
    h = ep.EpHandle(cfg_of(wl, dtype))
    h.layout(topk.cuda())
    R, H = wl.recv_capacity, wl.hidden
    if dtype == "fp8":
        recv = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
    else:
        recv = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
        scales = None
    rw = torch.full((R,), -3.0, device="cuda")
    ri = torch.full((R,), -9, dtype=torch.int32, device="cuda")
    h.dispatch(case["x"], recv, scales, w.cuda(), rw, ri)
    torch.cuda.synchronize()
    ref = ref_layout(wl, topk.numpy())
    want_w = np.full(R, -3.0, np.float32)
    want_i = np.full(R, -9, np.int32)
    oracle.forward_routing(topk.numpy(), w.numpy(), ref["dst_slot"], want_w, want_i)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), want_w.view(np.uint32))
    assert np.array_equal(ri.cpu().numpy(), want_i)
    # the rows themselves are unchanged by forwarding
    if dtype == "bf16":
        rx = np.zeros((R, H), np.uint16)
        oracle.dispatch_bf16(synth.bits16(case["x"]), ref["dst_slot"], rx)
        assert np.array_equal(synth.bits16(recv), rx)
    # only the ids are forwarded when only recv_topk_idx is given
    ri2 = torch.full((R,), -9, dtype=torch.int32, device="cuda")
    h.dispatch(case["x"], recv, scales, None, None, ri2)
    torch.cuda.synchronize()
    assert np.array_equal(ri2.cpu().numpy(), want_i)
    assert h.status() == 0


def test_handle_keeps_a_copy_of_the_ids():
    wl = synth.WORKLOADS["tiny"]
    topk = synth.gen_topk(wl, mask_frac=0.1)
    topk[2, 1] = wl.num_experts + 5          # out of range -> -1 in the copy
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    torch.cuda.synchronize()
    want = topk.numpy().astype(np.int32)
    want[(want < 0) | (want >= wl.num_experts)] = -1
    assert np.array_equal(h.field(ep.FIELD_TOPK_IDX).cpu().numpy(), want)
    assert h.status() == ep.ERR_BAD_EXPERT


def combine_inputs(wl, mask=0.0):
    topk = synth.gen_topk(wl, mask_frac=mask)
    ref = ref_layout(wl, topk.numpy())
    y = synth.gen_y(wl, valid_rows=ref["meta"][:, 0] >= 0, device="cuda")
    w = synth.gen_weights(wl)
    bias = synth.gen_bf16_normal(wl.num_tokens, wl.hidden, seed=wl.seed * 16 + 7, device="cuda")
    return topk, ref, y, w, bias


@pytest.mark.parametrize("name,use_bias,out_dtype,use_w", [
    ("tiny", True, "bf16", True), ("tiny", True, "fp32", True), ("tiny", False, "fp32", True),
    ("decode", True, "fp32", True), ("decode", True, "bf16", False),
    ("skewed", True, "bf16", True)])
def test_combine_ex_matches_the_oracle(name, use_bias, out_dtype, use_w):
    wl = synth.WORKLOADS[name]
    topk, ref, y, w, bias = combine_inputs(wl, 0.1 if name == "tiny" else 0.0)
    h = ep.EpHandle(cfg_of(wl, use_weights=use_w))
    h.layout(topk.cuda())
    dt = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    out = torch.full((wl.num_tokens, wl.hidden), -1, dtype=dt, device="cuda")
    h.combine(y, w.cuda() if use_w else None, out, bias if use_bias else None)
    torch.cuda.synchronize()
    want = oracle.combine_ex(synth.bits16(y), ref["dst_slot"], w.numpy() if use_w else None,
                             synth.bits16(bias) if use_bias else None, out_dtype)
    if out_dtype == "fp32":
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    else:
        assert np.array_equal(synth.bits16(out), want)


def test_combine_ex_sixteen_byte_aligned_buffers():
    wl = synth.WORKLOADS["tiny"]
    topk, ref, y, w, bias = combine_inputs(wl)
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    N, H = wl.num_tokens, wl.hidden
    base = torch.zeros(N * H + 8, dtype=torch.float32, device="cuda")
    out = base[4:4 + N * H].view(N, H)                 # 16- but not 32-byte aligned
    assert out.data_ptr() % 32 == 16
    h.combine(y, w.cuda(), out, bias)
    torch.cuda.synchronize()
    want = oracle.combine_ex(synth.bits16(y), ref["dst_slot"], w.numpy(), synth.bits16(bias), "fp32")
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_combine_ex_prefill_sampled():
    wl = synth.WORKLOADS["prefill_bf16"]
    topk, ref, y, w, bias = combine_inputs(wl)
    h = ep.EpHandle(cfg_of(wl))
    h.layout(topk.cuda())
    out = torch.empty((wl.num_tokens, wl.hidden), dtype=torch.float32, device="cuda")
    h.combine(y, w.cuda(), out, bias)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    sel = np.unique(np.concatenate([rng.choice(wl.num_tokens, 1500, replace=False),
                                    [0, wl.num_tokens - 1]]))
    ds = ref["dst_slot"][sel]
    rows = torch.from_numpy(ds.reshape(-1).astype(np.int64)).cuda()
    slots = np.arange(ds.size, dtype=np.int32).reshape(ds.shape)
    tsel = torch.from_numpy(sel).cuda()
    want = oracle.combine_ex(synth.bits16(y[rows]), slots, w.numpy()[sel], synth.bits16(bias[tsel]),
                             "fp32")
    assert np.array_equal(out[tsel].cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("name,dtype", [("tiny", "fp32"), ("tiny", "fp4x2"), ("decode", "fp32"),
                                        ("decode", "fp4x2"), ("skewed", "fp4x2")])
def test_opaque_transports_move_rows_unchanged(name, dtype):
    wl = synth.WORKLOADS[name]
    topk = synth.gen_topk(wl, mask_frac=0.05)
    row_bytes = 4 * wl.hidden if dtype == "fp32" else wl.hidden // 2
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randint(0, 256, (wl.num_tokens, row_bytes), dtype=torch.uint8, device="cuda",
                      generator=g)
    if dtype == "fp32":
        x = x.view(torch.float32)
    h = ep.EpHandle(cfg_of(wl, dtype))
    h.layout(topk.cuda())
    recv = torch.full((wl.recv_capacity, row_bytes), 0x5A, dtype=torch.uint8, device="cuda")
    h.dispatch(x, recv)
    torch.cuda.synchronize()
    ref = ref_layout(wl, topk.numpy())
    want = np.full((wl.recv_capacity, row_bytes), 0x5A, np.uint8)
    oracle.dispatch_bytes(x.view(torch.uint8).cpu().numpy(), ref["dst_slot"], want)
    assert np.array_equal(recv.cpu().numpy(), want)
    assert h.variant(1).startswith("ep_dispatch_" + dtype)


def test_shared_layout_feeds_other_dtypes_and_widths():
    # one layout (bf16 handle) serves an FP8 dispatch and a combine of another width
    wl = synth.WORKLOADS["decode"]
    case = synth.make_case(wl, device="cuda", mask_frac=0.05)
    h16 = ep.EpHandle(cfg_of(wl, "bf16"))
    h8 = ep.EpHandle(cfg_of(wl, "fp8"), layout_of=h16)
    wide = wl.with_(hidden=2 * wl.hidden)
    hw = ep.EpHandle(cfg_of(wide, "bf16", use_weights=False), layout_of=h8)   # shares h16's
    h16.layout(case["topk_idx"].cuda())
    ref = ref_layout(wl, case["topk_idx"].numpy())
    R, H = wl.recv_capacity, wl.hidden
    recv8 = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
    h8.dispatch(case["x"], recv8, scales)
    y = synth.gen_bf16_normal(R, 2 * H, seed=9, device="cuda")
    out = torch.empty((wl.num_tokens, 2 * H), dtype=torch.bfloat16, device="cuda")
    hw.combine(y, None, out)
    torch.cuda.synchronize()
    rq = np.zeros((R, H), np.uint8)
    rs = np.zeros((R, H // 128), np.float32)
    oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], rq, rs)
    assert np.array_equal(recv8.cpu().numpy(), rq)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(synth.bits16(out), oracle.combine(synth.bits16(y), ref["dst_slot"], None))
    for f in (ep.FIELD_DST_SLOT, ep.FIELD_RECV_SRC_METADATA, ep.FIELD_PSUM_PER_EXPERT):
        assert torch.equal(h8.field(f), h16.field(f)) and torch.equal(hw.field(f), h16.field(f))
    assert h8.variant(0) == h16.variant(0)
    assert h8.status() == 0
    # the shared handle computes no layout of its own
    with pytest.raises(ep.EpError) as e:
        h8.layout(case["topk_idx"].cuda())
    assert e.value.code == ep.EP_EINVAL
    # a new routing on the owner is what the shared handles see next
    topk2 = synth.gen_topk(wl.with_(seed=wl.seed + 5))
    h16.layout(topk2.cuda())
    h8.dispatch(case["x"], recv8, scales)
    torch.cuda.synchronize()
    ref2 = ref_layout(wl, topk2.numpy())
    rq2 = np.zeros((R, H), np.uint8)
    oracle.dispatch_fp8(synth.bits16(case["x"]), ref2["dst_slot"], rq2, np.zeros_like(rs))
    got = recv8.cpu().numpy()
    filled = ref2["meta"][:, 0] >= 0
    assert np.array_equal(got[filled], rq2[filled])


def test_shared_layout_rejects_a_different_routing_shape():
    wl = synth.WORKLOADS["tiny"]
    h = ep.EpHandle(cfg_of(wl))
    for bad in (wl.with_(topk=2), wl.with_(alignment=4), wl.with_(world_size=2, max_tok_per_rank=64)):
        with pytest.raises(ep.EpError) as e:
            ep.EpHandle(cfg_of(bad), layout_of=h)
        assert e.value.code == ep.EP_EINVAL
    ne = ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                     wl.topk, wl.alignment, "bf16", False, no_expand=True)
    with pytest.raises(ep.EpError):
        ep.EpHandle(ne, layout_of=h)


# The dispatch geometry table splits each row over two CTAs for batches of up to
# 2048 tokens; EP_GB300_DISPATCH_SLICES (read when the handle is built) pins the
# choice, so both geometries are checked on small and large batches.
@pytest.mark.parametrize("slices", ["1", "2"])
@pytest.mark.parametrize("name,dtype", [("decode", "bf16"), ("decode", "fp8"), ("skewed", "bf16"),
                                        ("tiny", "fp32"), ("tiny", "fp8")])
def test_dispatch_row_slices(name, dtype, slices, monkeypatch):
    monkeypatch.setenv("EP_GB300_DISPATCH_SLICES", slices)
    wl = synth.WORKLOADS[name]
    case = synth.make_case(wl, device="cuda", mask_frac=0.05)
    topk, w = case["topk_idx"], case["topk_weights"]
    h = ep.EpHandle(cfg_of(wl, dtype))
    h.layout(topk.cuda())
    ref = ref_layout(wl, topk.numpy())
    R, H = wl.recv_capacity, wl.hidden
    rw = torch.full((R,), -3.0, device="cuda")
    ri = torch.full((R,), -9, dtype=torch.int32, device="cuda")
    want_w = np.full(R, -3.0, np.float32)
    want_i = np.full(R, -9, np.int32)
    oracle.forward_routing(topk.numpy(), w.numpy(), ref["dst_slot"], want_w, want_i)
    if dtype == "fp8":
        recv = torch.zeros((R, H), dtype=torch.uint8, device="cuda")
        scales = torch.zeros((R, H // 128), dtype=torch.float32, device="cuda")
        h.dispatch(case["x"], recv, scales, w.cuda(), rw, ri)
        rq = np.zeros((R, H), np.uint8)
        rs = np.zeros((R, H // 128), np.float32)
        oracle.dispatch_fp8(synth.bits16(case["x"]), ref["dst_slot"], rq, rs)
        torch.cuda.synchronize()
        assert np.array_equal(recv.cpu().numpy(), rq)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    else:
        rb = 2 * H if dtype == "bf16" else 4 * H
        x = case["x"] if dtype == "bf16" else torch.randint(
            0, 256, (wl.num_tokens, rb), dtype=torch.uint8, device="cuda",
            generator=torch.Generator(device="cuda").manual_seed(4)).view(torch.float32)
        recv = torch.full((R, rb), 0x5A, dtype=torch.uint8, device="cuda")
        h.dispatch(x, recv.view(torch.bfloat16) if dtype == "bf16" else recv.view(torch.float32),
                   None, w.cuda(), rw, ri)
        want = np.full((R, rb), 0x5A, np.uint8)
        oracle.dispatch_bytes(x.contiguous().view(torch.uint8).cpu().numpy(), ref["dst_slot"], want)
        torch.cuda.synchronize()
        assert np.array_equal(recv.cpu().numpy(), want)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), want_w.view(np.uint32))
    assert np.array_equal(ri.cpu().numpy(), want_i)
    assert h.status() == 0
