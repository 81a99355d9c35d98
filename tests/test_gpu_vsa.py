"""GPU parity of block-sparse video attention (VSA) through the C ABI, against the fp64 oracle.

Selection (an integer decision taken from fp32 scores): the GPU's gate scores are compared with
the oracle's within a bound derived from fp32 accumulation; the GPU's selected set must be a
valid top-k of the oracle's scores up to that bound (blocks whose scores differ by less may be
taken in either order), and must equal the oracle's selection wherever the k-th and (k+1)-th
scores are further apart than the bound.  Attention: the oracle evaluates the fine attention on
the GPU's own selection (and on explicit selections), tolerances as for the other attention paths.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_REL = 2e-2, 2e-3, 1e-4


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


def _close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


def _lse_close(got, ref, what):
    rel = np.abs(np.asarray(got, np.float64) - ref) / np.maximum(np.abs(ref), 1.0)
    assert rel.max() <= LSE_REL, f"{what}: lse rel {rel.max():.3e}"


def _score_bound(q, k, grid, block, D):
    """Per-row bound on |fp32 score - fp64 score| for the GPU's accumulation: a block mean is a
    sequential fp32 sum of <= 64 rows times a rounded 1/count (error <= 65 u mean|x| per element),
    the score a D-term fp32 dot product (error <= D u sum |qm kd|) and one scaling; u = 2^-24.
    Doubled for margin; the row maximum is used for the whole row."""
    u = 2.0 ** -24
    qf, kf = q.float().numpy(), k.float().numpy()
    qm = np.abs(oracle.vsa_block_means(qf, grid, block))
    km = np.abs(oracle.vsa_block_means(kf, grid, block))
    qa = oracle.vsa_block_means(np.abs(qf), grid, block)
    ka = oracle.vsa_block_means(np.abs(kf), grid, block)
    kt = lambda x: np.transpose(x, (0, 2, 1))
    dot = np.matmul(qm, kt(km))
    means = np.matmul(qa, kt(km)) + np.matmul(qm, kt(ka))
    b = 2.0 * u / np.sqrt(D) * (D * dot + 65.0 * means) + u * dot / np.sqrt(D)
    return b.max(axis=2)   # [H, nblk]


def _check_selection(sel, scores_gpu, q, k, grid, block, topk, D, rows=None):
    ref = oracle.vsa_block_scores(q, k, grid, block)
    bound = _score_bound(q, k, grid, block, D)
    H, nblk, _ = ref.shape
    exact = 0
    for h in range(H):
        for a in (range(nblk) if rows is None else rows):
            b = bound[h, a]
            if scores_gpu is not None:
                assert np.abs(scores_gpu[h, a] - ref[h, a]).max() <= b, f"scores h{h} a{a}"
            ids = sel[h, a]
            assert len(ids) == topk and np.all(np.diff(ids) > 0) and ids[0] >= 0 and ids[-1] < nblk
            srt = np.sort(ref[h, a])[::-1]
            kth = srt[topk - 1]
            chosen = np.zeros(nblk, bool)
            chosen[ids] = True
            assert np.all(ref[h, a][chosen] >= kth - 2 * b), f"h{h} a{a}: a chosen block scores too low"
            assert np.all(ref[h, a][~chosen] <= kth + 2 * b), f"h{h} a{a}: a better block was left out"
            if topk == nblk or srt[topk - 1] - srt[topk] > 2 * b:
                assert np.array_equal(ids, oracle.vsa_select(ref[h:h + 1, a:a + 1], topk)[0, 0])
                exact += 1
    return exact


def _qkv(seed, n, H, D):
    rng = np.random.default_rng(seed)
    return [torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(torch.bfloat16)
            for _ in range(3)]


# grids: ragged blocks on every axis with 18 blocks (a tail item of two blocks), only full blocks
# (8), and 5 blocks (a tail item holding a single block)
GRIDS = [(5, 9, 11), (8, 8, 8), (4, 4, 20)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("grid", GRIDS)
def test_select_is_a_valid_top_k_of_the_oracle_scores(h3, dev, D, grid):
    n = grid[0] * grid[1] * grid[2]
    q, k, _ = _qkv(n + D, n, 3, D)
    nblk = oracle.vsa_block_count(grid, (4, 4, 4))
    for topk in sorted({1, min(3, nblk), nblk}):
        sel, scores = h3.vsa_select(q.to(dev), k.to(dev), grid, topk)
        torch.cuda.synchronize()
        assert h3.get_device_error(dev) == 0
        exact = _check_selection(sel.cpu().numpy(), scores.cpu().numpy(), q, k, grid, (4, 4, 4), topk, D)
        assert exact >= 3 * nblk // 2, f"too few rows with a clear top-k margin ({exact})"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("grid", GRIDS)
def test_attention_over_gpu_selection_matches_oracle(h3, dev, D, grid):
    n = grid[0] * grid[1] * grid[2]
    q, k, v = _qkv(7 * n + D, n, 3, D)
    nblk = oracle.vsa_block_count(grid, (4, 4, 4))
    for topk in sorted({1, min(3, nblk), nblk}):
        sel, _ = h3.vsa_select(q.to(dev), k.to(dev), grid, topk)
        o, lse = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, sel, return_lse=True)
        torch.cuda.synchronize()
        assert h3.get_device_error(dev) == 0
        ref_o, ref_lse = oracle.vsa_attention(q, k, v, grid, (4, 4, 4), sel.cpu().numpy())
        _close(o.float().cpu().numpy(), ref_o, f"vsa {grid} D {D} topk {topk}")
        _lse_close(lse.cpu().numpy(), ref_lse, f"vsa {grid} D {D} topk {topk}")


def test_full_selection_equals_dense_attention_and_self_selection_equals_block_windows(h3, dev):
    grid, D, H = (5, 9, 11), 128, 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = _qkv(11, n, H, D)
    nblk = oracle.vsa_block_count(grid, (4, 4, 4))
    full = torch.arange(nblk, dtype=torch.int32).repeat(H, nblk, 1).contiguous()
    o = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, full.to(dev))
    ref_o, _ = oracle.varlen_attention(q, k, v, [0, n])
    _close(o.float().cpu().numpy(), ref_o, "all blocks selected = dense attention")
    self_sel = torch.arange(nblk, dtype=torch.int32)[None, :, None].repeat(H, 1, 1).contiguous()
    o = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, self_sel.to(dev))
    wo = h3.window_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, (4, 4, 4), (0, 0, 0))
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    ref_o, _ = oracle.vsa_attention(q, k, v, grid, (4, 4, 4), self_sel.numpy())
    _close(o.float().cpu().numpy(), ref_o, "each block selects itself")
    _close(wo.float().cpu().numpy(), ref_o, "window attention with block-sized windows")


def test_random_explicit_selections_and_unselected_blocks_never_read(h3, dev):
    grid, D, H = (8, 8, 12), 128, 2   # 2 x 2 x 3 = 12 full blocks
    n = grid[0] * grid[1] * grid[2]
    q, k, v = _qkv(12, n, H, D)
    nblk = 12
    rng = np.random.default_rng(13)
    # every query block draws 4 of the blocks 0..9; blocks 10 and 11 are selected by nobody
    sel = np.stack([np.stack([np.sort(rng.choice(10, 4, replace=False)) for _ in range(nblk)])
                    for _ in range(H)]).astype(np.int32)
    o = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, torch.from_numpy(sel).to(dev))
    ref_o, _ = oracle.vsa_attention(q, k, v, grid, (4, 4, 4), sel)
    _close(o.float().cpu().numpy(), ref_o, "random selection")
    ids = oracle.vsa_block_ids(grid, (4, 4, 4))
    k2, v2 = k.clone(), v.clone()
    for b in (10, 11):
        k2[torch.from_numpy(ids == b)] = float("nan")
        v2[torch.from_numpy(ids == b)] = float("inf")
    o2 = h3.vsa_attn_fwd(q.to(dev), k2.to(dev), v2.to(dev), grid, torch.from_numpy(sel).to(dev))
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    assert torch.equal(o.cpu(), o2.cpu()), "an unselected block changed the output"
    # reversed list order: the same keys, the same result up to summation order
    o3 = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid,
                         torch.from_numpy(np.ascontiguousarray(sel[:, :, ::-1])).to(dev))
    _close(o3.float().cpu().numpy(), ref_o, "reversed selection lists")


def test_bad_block_index_is_reported_not_faulted(h3, dev):
    grid, D, H = (8, 8, 8), 64, 1
    n = 512
    q, k, v = _qkv(14, n, H, D)
    sel = torch.zeros((H, 8, 2), dtype=torch.int32)
    sel[:, :, 1] = 1
    sel[0, 3, 1] = 8          # one past the last block
    h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, sel.to(dev))
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 10   # H3_ERR_BAD_BLOCK_INDEX
    assert h3.get_device_error(dev) == 0


def test_video_grid_at_bench_size_sampled(h3, dev):
    """The 1344x768 latent (32x48x84, 2016 blocks), 24 heads x 128, top 252 (1/8), in the bench's
    launch configuration; selection and attention checked on sampled query blocks."""
    wl = W.vsa_video()
    grid, block, topk = wl.grid, wl.block, wl.topk
    q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
    sel, scores = h3.vsa_select(q, k, grid, topk)
    o, lse = h3.vsa_attn_fwd(q, k, v, grid, sel, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    nblk = oracle.vsa_block_count(grid, block)
    rng = np.random.default_rng(15)
    blocks = np.unique(np.concatenate([[0, 1, 2, 3, nblk - 1], rng.choice(nblk, 11, replace=False)]))
    heads = [0, 13, 23]
    sel_np = sel.cpu().numpy()[heads]
    qh, kh, vh = wl.q[:, heads], wl.k[:, heads], wl.v[:, heads]   # heads are independent
    exact = _check_selection(sel_np, scores.cpu().numpy()[heads], qh, kh, grid, block, topk,
                             wl.head_dim, rows=blocks)
    assert exact >= blocks.size  # N(0,1) inputs: the 252nd and 253rd scores are well apart
    ids = oracle.vsa_block_ids(grid, block)
    rows = np.nonzero(np.isin(ids, blocks))[0]
    ref_o, ref_lse = oracle.vsa_attention(qh, kh, vh, grid, block, sel_np, rows=rows)
    got = o.float().cpu().numpy()[:, heads]
    _close(got[rows], ref_o[rows], "vsa 32x48x84 sampled")
    _lse_close(lse.cpu().numpy()[heads][:, rows], ref_lse[:, rows], "vsa 32x48x84 sampled")


@pytest.mark.parametrize("block", [(2, 4, 8), (8, 2, 4)])
def test_non_cubic_64_token_blocks(h3, dev, block):
    """The block shape is the caller's as long as it holds 64 tokens: selection and attention
    with 2x4x8 and 8x2x4 blocks on a grid cropped on every axis."""
    grid, D, H = (9, 10, 13), 64, 2
    n = grid[0] * grid[1] * grid[2]
    q, k, v = _qkv(17 + block[0], n, H, D)
    nblk = oracle.vsa_block_count(grid, block)
    topk = min(4, nblk)
    sel, scores = h3.vsa_select(q.to(dev), k.to(dev), grid, topk, block=block)
    o, lse = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, sel, block=block, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    sel_np = sel.cpu().numpy()
    _check_selection(sel_np, scores.cpu().numpy(), q, k, grid, block, topk, D)
    ref_o, ref_lse = oracle.vsa_attention(q, k, v, grid, block, sel_np)
    _close(o.float().cpu().numpy(), ref_o, f"vsa block {block}")
    _lse_close(lse.cpu().numpy(), ref_lse, f"vsa block {block}")


def _schedule(ws, H, nblk, topk):
    """The key/value schedule in the attention's workspace: per (head, pair) the step list
    [topk, 2] of (block | use << 28) words, the step count and the shared-block count."""
    pairs = H * ((nblk + 1) // 2)
    raw = ws.cpu().numpy()
    off = (pairs * topk * 8 + 255) // 256 * 256
    steps = raw[:pairs * topk * 8].view(np.uint32).reshape(H, -1, topk, 2)
    counts = raw[off:off + pairs * 8].view(np.int32).reshape(H, -1, 2)
    return steps, counts[..., 0], counts[..., 1]


def _overlap_lists(case, nblk, topk, rng):
    """Selection lists [nblk, topk] whose paired query blocks (2p, 2p + 1) share a chosen number
    of blocks."""
    sel = np.zeros((nblk, topk), np.int32)
    for p in range(0, nblk, 2):
        a = np.sort(rng.choice(nblk, topk, replace=False))
        if case == "identical":
            b = a.copy()
        elif case == "disjoint":
            rest = np.setdiff1d(np.arange(nblk), a)
            b = np.sort(rng.choice(rest, topk, replace=False))
        elif case == "odd_overlap":       # 3 shared, the rest disjoint
            rest = np.setdiff1d(np.arange(nblk), a)
            b = np.sort(np.concatenate([a[:3], rng.choice(rest, topk - 3, replace=False)]))
        elif case == "repeats":           # sorted lists with repeated ids (each copy counts)
            a = np.sort(rng.choice(4, topk))
            b = np.sort(rng.choice(4, topk))
        elif case == "one_unsorted":      # pair 0's second list reversed: one step per entry there
            b = np.sort(rng.choice(nblk, topk, replace=False))
            if p == 0:
                b = b[::-1].copy()
        else:                             # random sorted lists
            b = np.sort(rng.choice(nblk, topk, replace=False))
        sel[p] = a
        if p + 1 < nblk:
            sel[p + 1] = b
    return sel


SCHEDULE_CASES = ["identical", "disjoint", "odd_overlap", "repeats", "one_unsorted", "random"]


@pytest.mark.parametrize("case", SCHEDULE_CASES)
@pytest.mark.parametrize("D", [64, 128])
def test_shared_blocks_schedule_against_oracle(h3, dev, case, D):
    """Paired query blocks that select the same key blocks share steps: the schedule in the
    workspace takes ceil(s/2) + topk - s steps for s shared selections of sorted lists (topk for
    unsorted ones), marks for each query block exactly its own list (as a multiset), and the
    attention over it equals the oracle's.  Grid 5x9x11: 18 blocks, ragged on every axis."""
    grid, H, topk = (5, 9, 11), 2, 6
    n = grid[0] * grid[1] * grid[2]
    nblk = oracle.vsa_block_count(grid, (4, 4, 4))
    rng = np.random.default_rng(100 * SCHEDULE_CASES.index(case) + D)
    sel = np.stack([_overlap_lists(case, nblk, topk, rng) for _ in range(H)])
    q, k, v = _qkv(21 + D, n, H, D)
    ws = torch.empty(h3.vsa_attn_workspace_size(grid, (4, 4, 4), H, topk), dtype=torch.uint8, device=dev)
    o, lse = h3.vsa_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, torch.from_numpy(sel).to(dev),
                             return_lse=True, workspace=ws)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    steps, nsteps, nshared = _schedule(ws, H, nblk, topk)
    for h in range(H):
        for p in range((nblk + 1) // 2):
            a, b = sel[h, 2 * p], sel[h, min(2 * p + 1, nblk - 1)]
            sorted_ = np.all(np.diff(a) >= 0) and np.all(np.diff(b) >= 0)
            shared = sum(min(np.count_nonzero(a == x), np.count_nonzero(b == x)) for x in np.unique(a))
            want = (shared + 1) // 2 + topk - shared if sorted_ else topk
            assert nsteps[h, p] == want, (case, h, p, nsteps[h, p], want)
            assert nshared[h, p] == (shared if sorted_ else 0)
            st = steps[h, p, :want]
            blk, use = st & ((1 << 28) - 1), st >> 28
            # the fixed layout the attention relies on: shared pairs, the odd shared block in
            # half 0, then each query block's own blocks in its own half
            s2 = nshared[h, p]
            lay = np.array([[3, 3]] * (s2 // 2) + [[3, 0]] * (s2 & 1) + [[1, 2]] * (want - (s2 + 1) // 2))
            assert np.array_equal(use, lay), (case, h, p)
            for qb, lst in ((0, a), (1, b)):
                mine = np.sort(blk[(use >> qb) & 1 == 1])
                assert np.array_equal(mine, np.sort(lst)), (case, h, p, qb)
            assert np.all(blk < nblk)
    ref_o, ref_lse = oracle.vsa_attention(q, k, v, grid, (4, 4, 4), sel)
    _close(o.float().cpu().numpy(), ref_o, f"schedule {case} D {D}")
    _lse_close(lse.cpu().numpy(), ref_lse, f"schedule {case} D {D}")


def test_shared_half_selection_at_bench_size_sampled(h3, dev):
    """The bench's fixed selection on the 1344x768 latent: paired query blocks share 126 of their
    252 blocks, so half of each pair's steps serve both halves of the tile.  Sampled query blocks
    of three heads against the oracle."""
    wl = W.vsa_video()
    grid, block, topk = wl.grid, wl.block, wl.topk
    nblk = oracle.vsa_block_count(grid, block)
    sel_np = W.vsa_paired_selection(9, wl.num_heads, nblk, topk, topk // 2)
    o, lse = h3.vsa_attn_fwd(wl.q.to(dev), wl.k.to(dev), wl.v.to(dev), grid,
                             torch.from_numpy(sel_np).to(dev), return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    rng = np.random.default_rng(16)
    blocks = np.unique(np.concatenate([[0, 1, 2, 3, nblk - 2, nblk - 1], rng.choice(nblk, 10, replace=False)]))
    heads = [0, 11, 23]
    ids = oracle.vsa_block_ids(grid, block)
    rows = np.nonzero(np.isin(ids, blocks))[0]
    ref_o, ref_lse = oracle.vsa_attention(wl.q[:, heads], wl.k[:, heads], wl.v[:, heads], grid, block,
                                          sel_np[heads], rows=rows)
    got = o.float().cpu().numpy()[:, heads]
    _close(got[rows], ref_o[rows], "vsa 32x48x84 shared-half sampled")
    _lse_close(lse.cpu().numpy()[heads][:, rows], ref_lse[:, rows], "vsa 32x48x84 shared-half sampled")
