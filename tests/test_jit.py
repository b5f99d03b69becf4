"""Run-time specialisation without a GPU: rendering, the SHA-256-keyed disk
cache with atomic publish, and cache hits ("MORI JIT v2" §1 and §3.4: the
configuration is the rendered text, the text is the cache key, entries are
published by a directory rename so racing processes agree).  Needs NVRTC;
skipped where it is missing."""
import hashlib
import os

import pytest
import torch.multiprocessing as mp

import __graft_entry__
import combine_ep_layout_gb300 as ep


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


@pytest.fixture()
def cache(tmp_path, monkeypatch):
    d = tmp_path / "jitcache"
    monkeypatch.setenv("EP_GB300_JIT_CACHE", str(d))
    return d


def precompile_or_skip(cfg):
    try:
        return ep.ep_jit_precompile(cfg)
    except ep.EpError as e:
        if e.code == ep.EP_EUNSUPPORTED:
            pytest.skip("NVRTC not available: " + str(e))
        raise


def entries(cache):
    root = cache / "sm_103a"
    return sorted(p.name for p in root.iterdir()) if root.exists() else []


def test_shape_outside_the_table_is_compiled_then_cached(cache):
    cfg = ep.make_cfg(4, 2560, 64, 8, 5, 1, "bf16", True)
    n, rep = precompile_or_skip(cfg)
    assert n == 2
    assert [l.split()[0] for l in rep] == ["ep_jit_dispatch_copy_rb5120_k5", "ep_jit_combine_w_h2560_k5"]
    assert all(" compiled " in l for l in rep)
    names = entries(cache)
    assert len(names) == 2
    for name in names:
        d = cache / "sm_103a" / name
        sig = (d / "signature.txt").read_bytes()
        # the directory carries the first 16 hex digits of SHA-256(signature)
        assert name.rsplit(".", 1)[1] == hashlib.sha256(sig).hexdigest()[:16]
        src = (d / "kernel.cu").read_text()
        assert src.encode() in sig and (d / "kernel.cubin").stat().st_size > 1000
        assert name.split(".")[1] in src          # the entry name is in the rendered text
    # a second request finds both in the cache
    n2, rep2 = precompile_or_skip(cfg)
    assert n2 == 0 and all(" cached " in l for l in rep2)
    assert entries(cache) == names


def test_each_configuration_gets_its_own_entry(cache):
    a = ep.make_cfg(4, 2560, 64, 8, 5, 1, "fp8", True)
    b = ep.make_cfg(4, 2560, 64, 8, 5, 1, "fp8", False)
    na, ra = precompile_or_skip(a)
    nb, rb = precompile_or_skip(b)
    assert na == 2 and nb == 1                     # the FP8 dispatch is shared
    assert ra[0].split()[0] == rb[0].split()[0] == "ep_jit_dispatch_fp8_h2560_k5"
    assert "cached" in rb[0]
    assert rb[1].split()[0] == "ep_jit_combine_h2560_k5"
    assert len(entries(cache)) == 3


def test_compiled_in_shapes_need_no_compilation(cache):
    cfg = ep.make_cfg(8, 7168, 4096, 32, 8, 128, "bf16", True)
    n, rep = precompile_or_skip(cfg)
    assert n == 0 and all("compiled-in" in l for l in rep)
    assert entries(cache) == []


def test_invalid_configuration_is_rejected(cache):
    with pytest.raises(ep.EpError) as e:
        ep.ep_jit_precompile(ep.make_cfg(4, 2564, 64, 8, 5, 1, "bf16", True))
    assert e.value.code == ep.EP_EINVAL


def _racer(cache_dir, q):
    os.environ["EP_GB300_JIT_CACHE"] = cache_dir
    import combine_ep_layout_gb300 as epm
    n, rep = epm.ep_jit_precompile(epm.make_cfg(4, 3584, 64, 8, 6, 1, "bf16", True))
    q.put((n, rep))


def test_racing_processes_publish_one_entry_each(tmp_path):
    probe = ep.make_cfg(4, 3584, 64, 8, 6, 1, "bf16", True)
    os.environ["EP_GB300_JIT_CACHE"] = str(tmp_path / "probe")
    try:
        precompile_or_skip(probe)
    finally:
        del os.environ["EP_GB300_JIT_CACHE"]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    d = str(tmp_path / "race")
    procs = [ctx.Process(target=_racer, args=(d, q)) for _ in range(3)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    results = [q.get(timeout=10) for _ in procs]
    assert all(len(rep) == 2 for _, rep in results)
    got = sorted(os.listdir(os.path.join(d, "sm_103a")))
    assert len(got) == 2                                 # one published entry per kernel
    assert os.listdir(os.path.join(d, "tmp")) == []      # losers removed their copies
