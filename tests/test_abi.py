"""CPU checks of the C boundary: the library loads, exports every function the
header declares, validates configurations on the host (no GPU needed), and the
compile-time config header compiles with a host-only compiler ("MORI JIT v2"
§3.5: the Cfg header needs no device compiler)."""
import ctypes
import os
import subprocess

import pytest

import __graft_entry__
import combine_ep_layout_gb300 as ep
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def test_exports_every_declared_symbol():
    names = ep.declared_symbols()
    assert len(names) == 15
    L = ep.load_library()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", ep._native.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(names) <= exported


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_recv_capacity_matches_the_oracle(name):
    wl = synth.WORKLOADS[name]
    cfg = ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                      wl.topk, wl.alignment, wl.dispatch_dtype, wl.use_weights)
    want = oracle.recv_capacity(wl.world_size * wl.max_tok_per_rank, wl.topk, wl.num_experts,
                                wl.alignment)
    assert ep.ep_recv_capacity(cfg) == want == wl.recv_capacity


BAD = [
    dict(world_size=0), dict(world_size=65), dict(max_tok_per_rank=0),
    dict(num_expert_per_rank=0), dict(num_expert_per_rank=257),  # E = 8*257 > 2048
    dict(num_expert_per_token=0), dict(num_expert_per_token=17),
    dict(expert_alignment=0), dict(expert_alignment=4097),
    dict(hidden_dim=7100), dict(hidden_dim=4), dict(hidden_dim=32776),
    dict(dispatch_dtype=2, hidden_dim=7176),   # FP8 needs hidden % 128 == 0
    dict(dispatch_dtype=9), dict(use_weights=2),
    dict(max_tok_per_rank=1 << 22),            # W*T > 2^24
    dict(no_expand=2),
    dict(no_expand=1, use_weights=1),          # rank rows are combined unweighted
]


@pytest.mark.parametrize("bad", BAD)
def test_invalid_configs_are_rejected_on_the_host(bad):
    base = dict(world_size=8, hidden_dim=7168, max_tok_per_rank=128, num_expert_per_rank=8,
                num_expert_per_token=8, expert_alignment=1, dispatch_dtype=0, use_weights=1)
    base.update(bad)
    cfg = ep.ep_cfg_t(**base)
    L = ep.load_library()
    h = ctypes.c_void_p()
    rc = L.ep_handle_create(ctypes.byref(cfg), ctypes.byref(h))
    assert rc == ep.EP_EINVAL
    assert h.value is None
    assert ep.ep_last_error()
    assert L.ep_recv_capacity(ctypes.byref(cfg)) == ep.EP_EINVAL


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_nonexpand_recv_capacity_matches_the_oracle(name):
    wl = synth.WORKLOADS[name]
    cfg = ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                      wl.topk, wl.alignment, wl.dispatch_dtype, False, no_expand=True)
    want = oracle.recv_capacity_nonexpand(wl.world_size * wl.max_tok_per_rank, wl.topk,
                                          wl.world_size)
    assert ep.ep_recv_capacity(cfg) == want == wl.world_size * wl.max_tok_per_rank * min(
        wl.topk, wl.world_size)


def test_noalloc_layout_refuses_the_nonexpand_layout():
    L = ep.load_library()
    cfg = ep.make_cfg(4, 1024, 32, 8, 4, 1, "bf16", False, no_expand=True)
    rc = L.ep_layout_noalloc(ctypes.byref(cfg), None, 0, None, None, None, None, None, None, None,
                             None, None)
    assert rc == ep.EP_EUNSUPPORTED
    assert "expand" in ep.ep_last_error()


def test_transport_dtypes_are_validated():
    L = ep.load_library()
    # fp32 and packed fp4 rows are served (capacity is answered without a GPU)
    for dt in (ep.EP_FP32, ep.EP_FP4X2):
        assert L.ep_recv_capacity(ctypes.byref(ep.make_cfg(8, 7168, 128, 8, 8, 1, dt, True))) > 0
    # an fp4 row must be a whole number of 16-byte units: hidden % 32 == 0
    bad = ep.make_cfg(8, 7176, 128, 8, 8, 1, ep.EP_FP4X2, True)
    h = ctypes.c_void_p()
    assert L.ep_handle_create(ctypes.byref(bad), ctypes.byref(h)) == ep.EP_EINVAL
    assert "FP4x2" in ep.ep_last_error()


def test_null_arguments_are_errors_not_crashes():
    L = ep.load_library()
    cfg = ep.make_cfg(4, 1024, 32, 8, 4)
    h = ctypes.c_void_p(1)
    assert L.ep_handle_create_shared(ctypes.byref(cfg), None, ctypes.byref(h)) == ep.EP_EINVAL
    assert h.value is None and "layout_src" in ep.ep_last_error()
    assert L.ep_handle_create(None, None) == ep.EP_EINVAL
    assert L.ep_layout(None, None, 0, None) == ep.EP_EINVAL
    assert L.ep_dispatch(None, None, None, None, None) == ep.EP_EINVAL
    assert L.ep_combine(None, None, None, None, None) == ep.EP_EINVAL
    L.ep_handle_free(None)
    assert L.ep_handle_status(None, None) == ep.EP_EINVAL


def test_cfg_header_compiles_without_a_device_compiler():
    inc = os.path.join(ROOT, "combine_ep_layout_gb300", "csrc")
    tu = '#include "ep_cfg.hpp"\nstatic_assert(epg::RecvCapacity(32768, 8, 256, 128) == 294656);\n' \
         'int main() { return epg::EpShapeFieldCount() == 4 ? 0 : 1; }\n'
    subprocess.run(["g++", "-std=c++20", "-fsyntax-only", "-Wall", "-Werror", "-I", inc, "-x", "c++",
                    "-"], input=tu, text=True, check=True)


def test_public_header_is_plain_c():
    tu = '#include "ep_gb300.h"\nint main(void) { ep_cfg_t c = {0}; return (int)sizeof c; }\n'
    subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-Wall", "-Werror", "-I",
                    os.path.join(ROOT, "include"), "-x", "c", "-"], input=tu, text=True, check=True)


def test_rank_magic_divides_exactly_over_the_whole_domain():
    """The layout divides expert ids by experts-per-rank with a multiply-high by
    floor(2^32/d) + 1; check the identity for every id < 2048 and d in [2, 2048]."""
    import numpy as np
    e = np.arange(2048, dtype=np.uint64)
    for d in range(2, 2049):
        m = np.uint64((1 << 32) // d + 1)
        assert np.array_equal((e * m) >> np.uint64(32), e // np.uint64(d)), d
