"""Pins of the oracle's FP8 path.

The format is OCP e4m3 ("fp8_ocp" = torch.float8_e4m3fn in the dtype table of
"MORI JIT Architecture"); per-128-channel fp32 scales travel with the token
("pack token data + sf", Dispatch data flow figure of "DeepEP overall
architecture analysis").  The pins are torch's own e4m3fn cast and decode
(a library routine, round-to-nearest-even, non-saturating), exhaustive
enumeration of codes and midpoints, and the e4m3 error bound.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_for_all_codes():
    mine = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = torch_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_encode_matches_torch_on_every_bf16_value_in_range():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float32)
    v = v[torch.isfinite(v) & (v.abs() <= 448)]
    for scale in (1.0, 3.0, 0.7, 2.0 ** -5, 1.0 / 448):
        w = (v * scale)
        w = w[w.abs() <= 448]
        ref = w.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = oracle.e4m3_encode(w.numpy())
        assert np.array_equal(got, ref), scale


def test_encode_matches_torch_on_random_fp32():
    g = torch.Generator().manual_seed(7)
    v = (torch.rand(1 << 20, generator=g) * 2 - 1) * 448
    v = torch.cat([v, torch.randn(1 << 18, generator=g) * 1e-3])
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v.numpy()), ref)


def test_midpoints_round_to_even():
    vals = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    for c in range(126):
        mid = (vals[c] + vals[c + 1]) / 2          # exact in fp32
        f = np.float32(mid)
        assert float(f) == mid
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([f]))[0] == want
        assert oracle.e4m3_encode(np.array([-f]))[0] == (0x80 | want)
        below = np.nextafter(f, np.float32(0))
        above = np.nextafter(f, np.float32(1000))
        assert oracle.e4m3_encode(np.array([below]))[0] == c
        assert oracle.e4m3_encode(np.array([above]))[0] == c + 1


def test_saturation_nan_and_zero():
    v = np.array([448, 449, 464, 465, 1e30, np.inf, -np.inf, -500, np.nan, 0.0, -0.0],
                 dtype=np.float32)
    got = oracle.e4m3_encode(v).tolist()
    assert got == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x00, 0x80]


def test_quant_row_scale_and_bound():
    wl = synth.WORKLOADS["prefill_fp8"]
    x = synth.gen_bf16_normal(64, wl.hidden, seed=123)
    bits = synth.bits16(x)
    xf = x.to(torch.float64).numpy()
    for r in range(bits.shape[0]):
        q, s = oracle.quant_fp8_row(bits[r])
        g = xf[r].reshape(-1, 128)
        amax = np.abs(g).max(axis=1)
        # s = amax / 448 in fp32
        assert np.array_equal(s, (amax.astype(np.float32) / np.float32(448)))
        deq = oracle.e4m3_decode(q).reshape(-1, 128)
        # the largest magnitude in each group maps to (close to) 448
        assert np.all(np.abs(deq).max(axis=1) >= 416)
        err = np.abs(deq * s[:, None].astype(np.float64) - g)
        bound = np.maximum(2.0 ** -4 * np.abs(g), 2.0 ** -10 * s[:, None]) * (1 + 2.0 ** -20) \
            + np.abs(g) * 2.0 ** -23
        assert np.all(err <= bound)


def test_quant_row_exact_power_of_two_group_hits_448():
    # amax a power of two: s = amax/448 and amax/s == 448 exactly -> code 0x7E
    row = torch.zeros(256, dtype=torch.float32)
    row[:128] = torch.linspace(-1, 1, 128)
    row[5] = -2.0
    row[128:] = 0.0
    row[200] = -0.0
    bits = synth.bits16(row.to(torch.bfloat16))
    q, s = oracle.quant_fp8_row(bits)
    assert s[0] == np.float32(2.0) / np.float32(448)
    assert q[5] == 0xFE
    assert s[1] == 0.0 and not q[128:].any()          # all-zero group


def test_negative_zero_in_nonzero_group():
    row = torch.zeros(128)
    row[0] = 1.0
    row[1] = -0.0
    q, s = oracle.quant_fp8_row(synth.bits16(row.to(torch.bfloat16)))
    assert q[1] == 0x80 and q[2] == 0x00 and q[0] == 0x7E


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_dispatch_fp8_writes_the_token_quantisation_to_each_slot(name):
    wl = synth.WORKLOADS[name].with_(dispatch_dtype="fp8")
    topk = synth.gen_topk(wl).numpy()
    x = synth.gen_x(wl)
    lay = oracle.layout(topk, wl.world_size, wl.max_tok_per_rank, wl.num_expert_per_rank,
                        wl.alignment)
    R, H = lay["rcap"], wl.hidden
    rx = np.full((R, H), 0xAB, np.uint8)
    rs = np.full((R, H // 128), -7.0, np.float32)
    bits = synth.bits16(x)
    oracle.dispatch_fp8(bits, lay["dst_slot"], rx, rs)
    written = np.zeros(R, bool)
    for t in range(wl.num_tokens):
        q, s = oracle.quant_fp8_row(bits[t])
        for k in range(wl.topk):
            r = lay["dst_slot"][t, k]
            assert np.array_equal(rx[r], q) and np.array_equal(rs[r], s)
            written[r] = True
    assert (rx[~written] == 0xAB).all() and (rs[~written] == -7.0).all()
