"""The allocation-free attention entry point (h3_varlen_attn_fwd_noalloc), called through the C ABI.

Some callers cannot allocate device memory -- their memory is owned by an external pool or
allocator, or a cudaMalloc there would stall or is not allowed -- so the library offers this
variant that keeps its work plan in a fixed array of its own.  It runs the same plan kernel and
the same attention kernel as h3_varlen_attn_fwd given a workspace that holds the plan alone (no
room to split the last wave), so on the same inputs its outputs must be the same bytes, call after
call: the shared array keeps the previous call's plan, which must never leak into the next one.

Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

NOALLOC_MAX_SEGMENTS = 16384  # H3_NOALLOC_MAX_SEGMENTS


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import packed_varlen_attention_modality_gb300 as h3

    return h3.load_library()


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _case(dev, wl):
    d = dict(q=wl.q.to(dev), k=wl.k.to(dev), v=wl.v.to(dev), cu=torch.from_numpy(wl.cu_seqlens).to(dev))
    d["C"], d["H"], d["D"] = wl.q.shape
    d["S"], d["maxs"] = wl.num_segments, max(1, wl.max_seqlen)
    d["N"] = wl.num_tokens
    return d


def _with_workspace(lib, dev, c):
    """The workspace entry point with the plan alone (the size returned for a max_seqlen below
    1024): like the no-alloc entry point, it then runs every work item whole."""
    o = torch.full_like(c["q"], 5.0)
    lse = torch.full((c["H"], c["C"]), 5.0, device=dev)
    nbytes = lib.h3_varlen_attn_workspace_size(c["S"], c["H"], 1, c["D"])
    ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=dev)
    st = lib.h3_varlen_attn_fwd(_p(c["q"]), _p(c["k"]), _p(c["v"]), _p(o), _p(lse), _p(c["cu"]), c["S"],
                                c["maxs"], c["C"], c["H"], c["D"], 0.0, _p(ws), nbytes, _stream(dev))
    assert st == 0
    return o, lse


def _no_alloc(lib, dev, c):
    o = torch.full_like(c["q"], 5.0)
    lse = torch.full((c["H"], c["C"]), 5.0, device=dev)
    st = lib.h3_varlen_attn_fwd_noalloc(_p(c["q"]), _p(c["k"]), _p(c["v"]), _p(o), _p(lse), _p(c["cu"]),
                                        c["S"], c["maxs"], c["C"], c["H"], c["D"], 0.0, _stream(dev))
    assert st == 0
    return o, lse


def _same(got, ref, N, what):
    """Same plan, same kernel, same inputs: the same bytes (pad rows untouched on both sides)."""
    o, lse = got
    o_ref, lse_ref = ref
    assert torch.equal(o, o_ref), f"{what}: output differs"
    assert torch.equal(lse, lse_ref), f"{what}: lse differs"
    assert torch.all(o[N:] == 5.0) and torch.all(lse[:, N:] == 5.0), what


def test_no_alloc_matches_workspace_entry_point_on_consecutive_calls(lib, dev):
    # each case follows one of another shape, so a plan left in the array by the previous call
    # (more segments, longer segments) would show if anything read it
    cases = [W.random_packed(31, [300, 1, 517, 0, 1024, 129], heads=4, head_dim=128, capacity=2048),
             W.tiny_example(capacity=64),
             W.random_packed(32, [256] * 40 + [77, 3], heads=2, head_dim=128, capacity=10400),
             W.random_packed(33, [2500, 40, 3], heads=3, head_dim=64, capacity=2600),
             W.tiny_example(capacity=64)]
    for wl in cases:
        c = _case(dev, wl)
        ref = _with_workspace(lib, dev, c)
        first = _no_alloc(lib, dev, c)
        second = _no_alloc(lib, dev, c)  # the array still holds the first call's plan
        torch.cuda.synchronize()
        assert lib.h3_get_device_error(_stream(dev)) == 0
        _same(first, ref, c["N"], f"{wl.name} first call")
        _same(second, ref, c["N"], f"{wl.name} second call")


def test_no_alloc_at_its_segment_limit(lib, dev):
    """Exactly H3_NOALLOC_MAX_SEGMENTS segments of 0-5 rows: the largest plan the array holds,
    and more segments than the plan orders longest-first (its unsorted branch)."""
    lengths = [int(x) for x in np.random.default_rng(34).integers(0, 6, NOALLOC_MAX_SEGMENTS)]
    wl = W.random_packed(34, lengths, heads=2, head_dim=64, capacity=sum(lengths) + 9)
    c = _case(dev, wl)
    assert c["S"] == NOALLOC_MAX_SEGMENTS
    ref = _with_workspace(lib, dev, c)
    for call in ("first", "second"):
        got = _no_alloc(lib, dev, c)
        torch.cuda.synchronize()
        assert lib.h3_get_device_error(_stream(dev)) == 0
        _same(got, ref, c["N"], f"{NOALLOC_MAX_SEGMENTS} segments, {call} call")


def test_no_alloc_refuses_more_segments_than_its_array_holds(lib, dev):
    limit = NOALLOC_MAX_SEGMENTS
    q = torch.zeros(64, 1, 64, dtype=torch.bfloat16, device=dev)
    cu = torch.zeros(limit + 2, dtype=torch.int32, device=dev)
    st = lib.h3_varlen_attn_fwd_noalloc(_p(q), _p(q), _p(q), _p(q), None, _p(cu), limit + 1, 1, 64, 1, 64,
                                        0.0, _stream(dev))
    assert st == 5  # H3_ERR_WORKSPACE, nothing launched
