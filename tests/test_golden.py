"""The oracle against the fixtures under tests/golden/: values derived by hand
from the pages' definitions (each file states its citation and derivation),
independent of both the oracle and the CUDA path."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    assert g["citation"] and g["derivation"]
    return g


def test_expand_layout_worked_example():
    g = load("layout_expand_worked_example.json")
    o = oracle.layout(np.array(g["topk_idx"], np.int64), g["world_size"], g["max_tok_per_rank"],
                      g["num_expert_per_rank"], g["alignment"])
    assert o["rcap"] == g["rcap"] and o["num_recv"] == g["num_recv"] and o["err"] == 0
    for k in ("cnt", "tok_per_rank", "psum_expert", "psum_rank", "dst_slot", "meta"):
        assert o[k].tolist() == g[k], k


def test_nonexpand_layout_worked_example():
    g = load("layout_nonexpand_worked_example.json")
    topk = np.array(g["topk_idx"], np.int64)
    o = oracle.layout_nonexpand(topk, g["world_size"], g["max_tok_per_rank"],
                                g["num_expert_per_rank"], g["alignment"])
    assert o["rcap"] == g["rcap"] and o["num_recv"] == g["num_recv"] and o["err"] == 0
    for k in ("cnt", "tok_per_rank", "psum_expert", "psum_rank", "dst_slot", "send_slot", "meta"):
        assert o[k].tolist() == g[k], k
    K = topk.shape[1]
    rw = np.full((g["rcap"], K), 9.0, np.float32)
    ri = np.full((g["rcap"], K), 9, np.int32)
    oracle.forward_routing_nonexpand(topk, np.array(g["topk_weights"], np.float32), o["dst_slot"],
                                     o["send_slot"], rw, ri)
    R = g["num_recv"]
    assert ri[:R].tolist() == g["recv_topk_idx_rows"]
    assert rw[:R].tolist() == g["recv_topk_weights_rows"]
    assert (ri[R:] == 9).all() and (rw[R:] == 9.0).all()


def test_e4m3_reference_points():
    g = load("e4m3_reference_points.json")
    vals = np.array([float(v) for v, _ in g["encode"]], np.float32)
    want = [int(c, 16) for _, c in g["encode"]]
    assert oracle.e4m3_encode(vals).tolist() == want
    codes = np.array([int(c, 16) for c, _ in g["decode"]], np.uint8)
    got = oracle.e4m3_decode(codes)
    for (c, v), x in zip(g["decode"], got):
        want_v = float(v)
        if math.isnan(want_v):
            assert math.isnan(x), c
        else:
            assert x == want_v and math.copysign(1.0, x) == math.copysign(1.0, want_v), c


@pytest.mark.parametrize("name", ["layout_expand_worked_example.json",
                                  "layout_nonexpand_worked_example.json",
                                  "e4m3_reference_points.json"])
def test_fixture_states_its_source(name):
    g = load(name)
    assert "'" in g["citation"] or "OCP" in g["citation"]
