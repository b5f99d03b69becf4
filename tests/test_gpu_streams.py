"""The handle calls that wait (ep_handle_create, ep_handle_status) wait for
their own work only, never for an unrelated busy stream.

A serving process keeps several streams busy; creating a handle for a new
configuration, or reading a handle's error word, must not stall them.  Here a
second stream runs a fixed-length device sleep (torch.cuda._sleep, a bounded
clock spin of tens of milliseconds) while the handle calls run; each call must
return while that stream is still busy.
"""
import time

import pytest
import torch

import combine_ep_layout_gb300 as ep
import synth

pytestmark = pytest.mark.gpu

SLEEP_CYCLES = 150_000_000   # ~75 ms at 2 GHz, ~150 ms at 1 GHz: bounded either way


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def cfg_of(wl):
    return ep.make_cfg(wl.world_size, wl.hidden, wl.max_tok_per_rank, wl.num_expert_per_rank,
                       wl.topk, wl.alignment, wl.dispatch_dtype, wl.use_weights)


def busy_stream():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES)
    return s


def test_handle_create_does_not_wait_for_other_streams():
    wl = synth.WORKLOADS["decode"]
    # the first handle of a configuration loads its kernels (module loading may
    # synchronise the context), so make one before the busy stream starts
    ep.EpHandle(cfg_of(wl)).free()
    torch.cuda.synchronize()
    s = busy_stream()
    t0 = time.perf_counter()
    h = ep.EpHandle(cfg_of(wl))
    dt = time.perf_counter() - t0
    still_busy = not s.query()
    s.synchronize()
    assert still_busy, "ep_handle_create returned only after the unrelated stream finished"
    assert dt < 0.03, dt
    # the new handle works (its metadata block was cleared before create returned)
    topk = synth.gen_topk(wl).cuda()
    h.layout(topk)
    assert h.status() == 0
    h.free()


def test_handle_status_waits_for_its_own_stream_only():
    wl = synth.WORKLOADS["tiny"]
    h = ep.EpHandle(cfg_of(wl))
    mine = torch.cuda.Stream()
    topk = synth.gen_topk(wl).cuda()
    h.layout(topk, stream=mine)
    torch.cuda.synchronize()
    s = busy_stream()
    h.layout(topk, stream=mine)
    assert h.status() == 0
    still_busy = not s.query()
    s.synchronize()
    assert still_busy, "ep_handle_status waited for an unrelated stream"
    h.free()
