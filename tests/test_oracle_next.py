"""Pins of the oracle's wider routines: opaque-payload dispatch (fp32 and packed
fp4 transports, "MORI JIT v2" §3.7), forwarding of the routing with each
received row (dispatch copy epilogue of "DeepEP overall architecture
analysis"), and combine with a bias and an fp32 output ("Combine data flow":
reduce weighted by topk_weights, "+ bias")."""
import numpy as np
import torch

import oracle
import synth


def lay(wl, mask_frac=0.0):
    topk = synth.gen_topk(wl, mask_frac=mask_frac).numpy()
    return topk, oracle.layout(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                               wl.alignment)


def test_bytes_dispatch_moves_rows_unchanged():
    wl = synth.WORKLOADS["tiny"].with_(alignment=4)
    topk, L = lay(wl, 0.1)
    rng = np.random.default_rng(0)
    for row_bytes in (4 * wl.hidden, wl.hidden // 2, 48):
        x = rng.integers(0, 256, size=(wl.num_tokens, row_bytes), dtype=np.uint8)
        recv = np.full((L["rcap"], row_bytes), 0x5A, np.uint8)
        oracle.dispatch_bytes(x, L["dst_slot"], recv)
        t, k = np.nonzero(L["dst_slot"] >= 0)
        assert np.array_equal(recv[L["dst_slot"][t, k]], x[t])
        untouched = np.ones(L["rcap"], bool)
        untouched[L["dst_slot"][t, k]] = False
        assert (recv[untouched] == 0x5A).all()


def test_bytes_dispatch_agrees_with_the_bf16_dispatch():
    wl = synth.WORKLOADS["decode"]
    topk, L = lay(wl)
    x = synth.bits16(synth.gen_x(wl))
    a = np.zeros((L["rcap"], wl.hidden), np.uint16)
    oracle.dispatch_bf16(x, L["dst_slot"], a)
    b = np.zeros((L["rcap"], 2 * wl.hidden), np.uint8)
    oracle.dispatch_bytes(x.view(np.uint8), L["dst_slot"], b)
    assert np.array_equal(a.view(np.uint8), b)


def test_forwarded_routing_follows_the_expert_segments():
    wl = synth.WORKLOADS["skewed"].with_(num_tokens=3000)
    topk, L = lay(wl, 0.05)
    w = synth.gen_weights(wl).numpy()
    rw = np.full(L["rcap"], -1.0, np.float32)
    ri = np.full(L["rcap"], -7, np.int32)
    oracle.forward_routing(topk, w, L["dst_slot"], rw, ri)
    # every filled row of expert e's segment carries e; padding rows untouched
    for e in range(wl.num_experts):
        a, n, b = L["psum_expert"][e], L["cnt"][e], L["psum_expert"][e + 1]
        assert (ri[a:a + n] == e).all()
        assert (ri[a + n:b] == -7).all()
    # the weights of a token's rows are its weights, in k order
    for t in range(0, wl.num_tokens, 97):
        for k in range(wl.topk):
            s = L["dst_slot"][t, k]
            if s >= 0:
                assert rw[s] == w[t, k]
    # total weight is conserved over the received rows
    assert np.isclose(rw[ri >= 0].astype(np.float64).sum(),
                      w[topk >= 0].astype(np.float64).sum())


def test_combine_ex_without_bias_is_combine():
    wl = synth.WORKLOADS["tiny"]
    topk, L = lay(wl, 0.1)
    y = synth.bits16(synth.gen_bf16_normal(L["rcap"], wl.hidden, seed=4))
    w = synth.gen_weights(wl).numpy()
    assert np.array_equal(oracle.combine_ex(y, L["dst_slot"], w), oracle.combine(y, L["dst_slot"], w))


def test_combine_ex_fp32_identity_experts_is_k_times_x_exactly():
    wl = synth.WORKLOADS["decode"]
    topk, L = lay(wl)
    x = synth.gen_x(wl)
    rx = np.zeros((L["rcap"], wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(x), L["dst_slot"], rx)
    out = oracle.combine_ex(rx, L["dst_slot"], None, None, "fp32")
    assert np.array_equal(out, (x.float() * wl.topk).numpy())


def test_combine_ex_bias_cancels_exactly():
    # identity experts, unit weights: the fold is K*x exactly; a bias of -K*x
    # (exact in bf16 for K a power of two) leaves +0.0 everywhere.
    wl = synth.WORKLOADS["tiny"]
    topk, L = lay(wl)
    x = synth.gen_x(wl)
    rx = np.zeros((L["rcap"], wl.hidden), np.uint16)
    oracle.dispatch_bf16(synth.bits16(x), L["dst_slot"], rx)
    bias = synth.bits16((-x.float() * wl.topk).to(torch.bfloat16))
    out = oracle.combine_ex(rx, L["dst_slot"], None, bias, "bf16")
    assert (out == 0).all()
    out32 = oracle.combine_ex(rx, L["dst_slot"], None, bias, "fp32")
    assert (out32.view(np.uint32) == 0).all()


def test_combine_ex_adds_the_bias_after_the_fold():
    # rows 2^24 and -2^24, bias 1: after the fold (0) + 1 = 1; a bias folded in
    # first would be absorbed: (1 + 2^24) rounds to 2^24, then - 2^24 = 0.
    y = synth.bits16(torch.tensor([[2.0 ** 24], [-(2.0 ** 24)]]).to(torch.bfloat16))
    slot = np.array([[0, 1]], np.int32)
    bias = synth.bits16(torch.tensor([[1.0]]).to(torch.bfloat16))
    assert oracle.combine_ex(y, slot, None, bias, "fp32")[0, 0] == 1.0


def test_combine_ex_fp32_within_the_fp64_bound():
    wl = synth.WORKLOADS["tiny"]
    topk, L = lay(wl)
    y = synth.gen_bf16_normal(L["rcap"], wl.hidden, seed=8)
    b = synth.gen_bf16_normal(wl.num_tokens, wl.hidden, seed=9)
    w = synth.gen_weights(wl).numpy()
    out = oracle.combine_ex(synth.bits16(y), L["dst_slot"], w, synth.bits16(b), "fp32")
    yf, bf = y.double().numpy(), b.double().numpy()
    exact = np.einsum("tk,tkh->th", w.astype(np.float64), yf[L["dst_slot"]]) + bf
    absum = np.einsum("tk,tkh->th", np.abs(w.astype(np.float64)), np.abs(yf[L["dst_slot"]])) + \
        np.abs(bf)
    assert np.all(np.abs(out - exact) <= (wl.topk + 1) * 2.0 ** -23 * absum + 1e-30)
