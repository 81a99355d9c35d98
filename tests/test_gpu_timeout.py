"""The attention kernels' bounded waits, made to run out on purpose (through the C ABI).

Every wait between the warps of an attention kernel gives up after a limit (2 s by default)
instead of spinning forever.  Here the key/value loader of every CTA is told to stop after three
tiles (h3_debug_stall_loads), as if it had stalled, and the limit is shortened to 20 ms
(h3_set_wait_limit_ns), so the waits of the warps that consume those tiles run out in the middle
of an otherwise valid launch.  Each variant (packed segments, windows in place, block-sparse)
must then:
  * end (the synchronise returns) and record H3_ERR_TIMEOUT in the error word;
  * make every later launch leave at once while that error is recorded (outputs untouched);
  * after h3_get_device_error() clears it, give the very bytes of a launch made before the
    timeout -- so no copy was left landing, no tensor memory was left allocated and no barrier
    state carried over.
Nothing here faults or hangs the GPU: no load is issued that would not be issued normally, what
the unwinding kernels wait for (copies and matrix products already issued) completes by itself,
and every other wait ends by its limit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

TIMEOUT = 7  # H3_ERR_TIMEOUT


@pytest.fixture(scope="module")
def h3():
    import __graft_entry__

    __graft_entry__.build()
    import packed_varlen_attention_modality_gb300 as h3

    h3.load_library()
    return h3


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def _timeout_then_recover(h3, dev, run, shape_o, shape_lse):
    """run(out, lse) launches one attention call into the given buffers."""
    assert h3.get_device_error(dev) == 0
    ref_o = torch.full(shape_o, 5.0, dtype=torch.bfloat16, device=dev)
    ref_l = torch.full(shape_lse, 5.0, dtype=torch.float32, device=dev)
    run(ref_o, ref_l)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    h3.set_wait_limit_ns(20_000_000)
    h3.debug_stall_loads(3)
    try:
        run(torch.empty(shape_o, dtype=torch.bfloat16, device=dev),
            torch.empty(shape_lse, dtype=torch.float32, device=dev))
        torch.cuda.synchronize()  # the launch ends although its waits ran out
        # the timeout is still recorded: a later launch leaves before touching anything
        o2 = torch.full(shape_o, 7.0, dtype=torch.bfloat16, device=dev)
        l2 = torch.full(shape_lse, 7.0, dtype=torch.float32, device=dev)
        run(o2, l2)
        torch.cuda.synchronize()
    finally:
        h3.debug_stall_loads(-1)
        h3.set_wait_limit_ns(0)
    assert torch.all(o2 == 7.0) and torch.all(l2 == 7.0)
    assert h3.get_device_error(dev) == TIMEOUT
    assert h3.get_device_error(dev) == 0
    o3 = torch.full(shape_o, 5.0, dtype=torch.bfloat16, device=dev)
    l3 = torch.full(shape_lse, 5.0, dtype=torch.float32, device=dev)
    run(o3, l3)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    assert torch.equal(o3, ref_o) and torch.equal(l3, ref_l)
    return o3, l3


@pytest.mark.parametrize("lengths,heads", [([4096, 300, 17], 8),  # 152 whole items: no split
                                           ([8192], 2)])            # every item split and merged
def test_packed_attention_timeout_unwinds(h3, dev, lengths, heads):
    wl = W.random_packed(61, lengths, heads=heads, head_dim=128, capacity=sum(lengths) + 67)
    q, k, v = (t.to(dev) for t in (wl.q, wl.k, wl.v))
    cu = torch.from_numpy(wl.cu_seqlens).to(dev)
    C, H, D = q.shape

    def run(o, lse):
        h3.varlen_attn_fwd(q, k, v, cu, wl.max_seqlen, out=o, lse=lse)

    o, lse = _timeout_then_recover(h3, dev, run, (C, H, D), (H, C))
    # and the recovered output is the attention: the short segments in full, a sample of the
    # long one's rows, against the oracle
    N = wl.num_tokens
    a = int(wl.cu_seqlens[1])
    rows = np.unique(np.r_[np.arange(0, a, 37), a - 1, np.arange(a, N)])
    ref, _ = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens, rows=rows)
    err = np.abs(o[rows].float().cpu().numpy() - ref[rows])
    assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_window_attention_timeout_unwinds(h3, dev):
    grid, win, shift = (16, 32, 32), (4, 8, 8), (2, 4, 4)
    n = grid[0] * grid[1] * grid[2]
    g = torch.Generator().manual_seed(62)
    q, k, v = (torch.randn((n, 8, 128), generator=g).to(torch.bfloat16).to(dev) for _ in range(3))

    def run(o, lse):
        h3.window_attn_fwd(q, k, v, grid, win, shift, out=o, lse=lse)

    _timeout_then_recover(h3, dev, run, (n, 8, 128), (8, n))


def test_vsa_attention_timeout_unwinds(h3, dev):
    grid, block, topk = (16, 16, 32), (4, 4, 4), 16
    n = grid[0] * grid[1] * grid[2]
    g = torch.Generator().manual_seed(63)
    q, k, v = (torch.randn((n, 4, 128), generator=g).to(torch.bfloat16).to(dev) for _ in range(3))
    nblk = h3.vsa_block_count(grid, block)
    rng = np.random.default_rng(63)
    sel = np.sort(np.stack([np.stack([rng.choice(nblk, topk, replace=False) for _ in range(nblk)])
                            for _ in range(4)]), axis=2).astype(np.int32)
    sel_d = torch.from_numpy(sel).to(dev)
    ws = torch.empty(h3.vsa_attn_workspace_size(grid, block, 4, topk), dtype=torch.uint8, device=dev)

    def run(o, lse):
        h3.vsa_attn_fwd(q, k, v, grid, sel_d, block=block, out=o, lse=lse, workspace=ws)

    _timeout_then_recover(h3, dev, run, (n, 4, 128), (4, n))
