"""Pins of the oracle's dispatch (bf16) and combine.

Dispatch moves bytes ("MORI JIT v2" §3.7: dtype is a transport property), so
it is pinned by byte equality.  Combine is the weighted reduce of the
"Combine data flow" figure of "DeepEP overall architecture analysis"; it is
pinned by the identity-expert round trip ("MORI JIT v2" §4 / §10: dispatch ->
identity expert -> combine), crafted inputs that fix the fma and the k order,
and an fp64 brute-force bound.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def layout_of(wl, mask_frac=0.0):
    topk = synth.gen_topk(wl, mask_frac=mask_frac).numpy()
    return topk, oracle.layout(topk, wl.world_size, wl.max_tok_per_rank,
                               wl.num_expert_per_rank, wl.alignment)


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_dispatch_bf16_is_a_byte_copy(name):
    wl = synth.WORKLOADS[name]
    if name == "skewed":
        wl = wl.with_(num_tokens=2048)
    topk, lay = layout_of(wl, mask_frac=0.05)
    x = synth.bits16(synth.gen_x(wl))
    rx = np.full((lay["rcap"], wl.hidden), 0xDEAD, np.uint16)
    oracle.dispatch_bf16(x, lay["dst_slot"], rx)
    t, k = np.nonzero(lay["dst_slot"] >= 0)
    rows = lay["dst_slot"][t, k]
    assert np.array_equal(rx[rows], x[t])
    untouched = np.ones(lay["rcap"], bool)
    untouched[rows] = False
    assert (rx[untouched] == 0xDEAD).all()


def bf16_of(a32):
    return torch.from_numpy(np.ascontiguousarray(a32, np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("name", ["tiny", "decode", "skewed"])
def test_identity_experts_unit_weights_give_k_times_x(name):
    wl = synth.WORKLOADS[name]
    if name == "skewed":
        wl = wl.with_(num_tokens=1024)
    topk, lay = layout_of(wl)
    x = synth.gen_x(wl)
    rx = np.zeros((lay["rcap"], wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(x), lay["dst_slot"], rx)
    out = oracle.combine(rx, lay["dst_slot"], None)
    # K*x is exact in fp32 (8-bit significand times K <= 8), so the only rounding
    # is the final one to bf16, which torch performs here.
    want = synth.bits16((x.to(torch.float32) * wl.topk).to(torch.bfloat16))
    assert np.array_equal(out, want)
    ones = np.ones((wl.num_tokens, wl.topk), np.float32)
    assert np.array_equal(oracle.combine(rx, lay["dst_slot"], ones), want)


def test_identity_experts_softmax_weights_give_x_back():
    wl = synth.WORKLOADS["decode"]
    topk, lay = layout_of(wl)
    x = synth.gen_x(wl)
    w = synth.gen_weights(wl).numpy()
    rx = np.zeros((lay["rcap"], wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(x), lay["dst_slot"], rx)
    out = torch.from_numpy(oracle.combine(rx, lay["dst_slot"], w).view(np.int16)).view(
        torch.bfloat16).to(torch.float64)
    xf = x.to(torch.float64)
    wsum = torch.from_numpy(w.astype(np.float64)).sum(1, keepdim=True)
    # out = bf16(fp32 sum of w_k*x) with sum_k w_k = 1 up to fp32 rounding
    err = (out - xf * wsum).abs()
    assert torch.all(err <= xf.abs() * (2.0 ** -8 + 16 * 2.0 ** -24) + 1e-30)


def test_k_order_is_ascending():
    # y rows: 2^24, 1, -2^24 (all exact in bf16), unit weights.
    # ascending: (2^24 + 1) rounds to 2^24 (tie to even), then - 2^24 -> 0.
    # descending would give (-2^24 + 1) + 2^24 = 1.
    y = synth.bits16(bf16_of(np.array([[2.0 ** 24], [1.0], [-2.0 ** 24]])))
    slot = np.array([[0, 1, 2]], np.int32)
    assert oracle.combine(y, slot, None)[0, 0] == 0x0000
    rev = np.array([[2, 1, 0]], np.int32)
    assert oracle.combine(y, rev, None)[0, 0] == synth.bits16(bf16_of(np.array([1.0])))[0]


def test_fused_multiply_add_not_multiply_then_add():
    # acc = w0*y0 = -(1 + 2^-7 + 2^-23); then w1*y1 = (1 + 2^-23)(1 + 2^-7)
    # = 1 + 2^-7 + 2^-23 + 2^-30, which needs 31 significant bits.  A fused
    # multiply-add keeps the 2^-30 term; rounding the product to fp32 first
    # loses it and the sum is 0.  Expected values computed exactly in fp64.
    w = np.array([[-(1 + 2.0 ** -7 + 2.0 ** -23), 1 + 2.0 ** -23]], np.float32)
    y_vals = np.array([[1.0], [1.0 + 2.0 ** -7]])                   # bf16-exact
    y = synth.bits16(bf16_of(y_vals))
    slot = np.array([[0, 1]], np.int32)
    acc = np.float32(np.float64(w[0, 0]) * y_vals[0, 0])
    exact = np.float64(w[0, 1]) * y_vals[1, 0] + np.float64(acc)    # exact in fp64
    fma = np.float32(exact)
    unfused = np.float32(np.float32(np.float64(w[0, 1]) * y_vals[1, 0]) + acc)
    assert fma == np.float32(2.0 ** -30) and unfused == 0
    got = oracle.combine(y, slot, w)[0, 0]
    assert got == oracle.f32_to_bf16(np.array([fma]))[0] == 0x3080


def test_masked_entries_contribute_nothing():
    y = synth.bits16(bf16_of(np.array([[1.5], [np.nan], [2.0]])))
    slot = np.array([[0, -1, 2]], np.int32)
    out = oracle.combine(y, slot, np.array([[1.0, 5.0, 0.5]], np.float32))
    assert out[0, 0] == synth.bits16(bf16_of(np.array([2.5])))[0]


def test_fp64_bound_on_random_experts():
    wl = synth.WORKLOADS["tiny"]
    topk, lay = layout_of(wl)
    y = synth.gen_bf16_normal(lay["rcap"], wl.hidden, seed=99)
    w = synth.gen_weights(wl).numpy()
    out = oracle.combine(synth.bits16(y), lay["dst_slot"], w)
    yf = y.to(torch.float64).numpy()
    exact = np.einsum("tk,tkh->th", w.astype(np.float64), yf[lay["dst_slot"]])
    absum = np.einsum("tk,tkh->th", np.abs(w.astype(np.float64)), np.abs(yf[lay["dst_slot"]]))
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    # fp32 fold error <= K * 2^-24 * sum|w y| (plus the products' rounding), then
    # one bf16 rounding <= 2^-9 relative.
    bound = wl.topk * 2.0 ** -23 * absum + np.abs(exact) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(got - exact) <= bound)
    # The final bf16 rounding alone is ~2^-9/sqrt(3) ~ 1.1e-3 relative L2 against
    # the exact sum, so the 1e-3 relative-L2 tolerance applies between an
    # implementation and this oracle (same bf16 output), not against fp64.
    assert np.abs(got - exact).max() <= 1e-2


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(3)
    v = torch.cat([torch.randn(1 << 20, generator=g) * 100,
                   torch.tensor([0.0, -0.0, 3.0e38, -3.4e38, 1e-40, float("inf")])])
    want = synth.bits16(v.to(torch.bfloat16))
    assert np.array_equal(oracle.f32_to_bf16(v.numpy()), want)
