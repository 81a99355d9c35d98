"""Pins for the block-sparse video attention (VSA) oracle, no GPU.

Each test ties oracle/vsa.py to something other than itself: closed-form block counts and sizes,
brute-force loops over coordinates, constructed inputs whose selection is known in advance, the
already-pinned dense and window attention routines, and a pure-Python masked softmax.
Source: [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section
"VSA: block-sparse attention" (4x4x4 = 64-token blocks, block-level gated scoring, top-k
selection, token-level attention between the selected blocks).
"""
import math

import numpy as np
import pytest

import oracle


def _normal(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("grid,counts", [((29, 40, 50), (8, 10, 13)), ((32, 48, 84), (8, 12, 21)),
                                         ((4, 4, 4), (1, 1, 1)), ((5, 9, 11), (2, 3, 3))])
def test_block_counts_closed_form(grid, counts):
    assert oracle.vsa_block_counts(grid, (4, 4, 4)) == counts
    assert oracle.vsa_block_count(grid, (4, 4, 4)) == counts[0] * counts[1] * counts[2]


@pytest.mark.parametrize("grid", [(29, 40, 50), (5, 9, 11)])
def test_block_sizes_factor_per_axis(grid):
    # an axis of length L cut in 4s has sizes 4, ..., 4, L - 4 * (ceil(L/4) - 1)
    ids = oracle.vsa_block_ids(grid, (4, 4, 4))
    sizes = np.bincount(ids)
    axes = [[min(4, L - 4 * i) for i in range((L + 3) // 4)] for L in grid]
    expect = np.einsum("i,j,k->ijk", *[np.array(a) for a in axes]).reshape(-1)
    assert np.array_equal(sizes, expect)
    assert sizes.sum() == grid[0] * grid[1] * grid[2]
    # 29 x 40 x 50: 7*10*12 interior blocks hold 64 tokens
    if grid == (29, 40, 50):
        assert int((sizes == 64).sum()) == 7 * 10 * 12


def test_block_ids_match_coordinate_loop():
    grid, block = (5, 6, 7), (2, 4, 3)
    ids = oracle.vsa_block_ids(grid, block)
    nh, nw = (6 + 3) // 4, (7 + 2) // 3
    n = 0
    for t in range(5):
        for h in range(6):
            for w in range(7):
                assert ids[n] == ((t // 2) * nh + h // 4) * nw + w // 3
                n += 1


def test_block_means_match_loop_and_constants():
    grid, block = (3, 5, 6), (2, 2, 4)
    x = _normal(1, (90, 2, 3))
    means = oracle.vsa_block_means(x, grid, block)
    ids = oracle.vsa_block_ids(grid, block)
    for b in range(oracle.vsa_block_count(grid, block)):
        rows = [i for i in range(90) if ids[i] == b]
        for h in range(2):
            for d in range(3):
                assert means[h, b, d] == pytest.approx(math.fsum(x[i, h, d] for i in rows) / len(rows),
                                                       rel=1e-14, abs=1e-15)
    # a block filled with one constant has that constant as its mean, exactly
    c = np.arange(oracle.vsa_block_count(grid, block), dtype=np.float64) * 0.25 - 1.0
    xc = np.repeat(c[ids][:, None, None], 2, axis=1).repeat(3, axis=2)
    assert np.array_equal(oracle.vsa_block_means(xc, grid, block)[0, :, 0], c)


def test_scores_from_rank_one_blocks_are_closed_form_and_not_transposed():
    # q rows of block a = alpha_a * u, k rows of block b = beta_b * u -> score = scale*alpha_a*beta_b*|u|^2
    grid, block = (4, 8, 8), (4, 4, 4)
    nblk = oracle.vsa_block_count(grid, block)          # 1 x 2 x 2 = 4
    ids = oracle.vsa_block_ids(grid, block)
    u = np.array([0.5, -1.0, 2.0, 0.25])
    alpha = np.array([1.0, -2.0, 0.5, 3.0])
    beta = np.array([-1.0, 4.0, 2.0, 0.5])
    q = (alpha[ids][:, None] * u)[:, None, :]
    k = (beta[ids][:, None] * u)[:, None, :]
    s = oracle.vsa_block_scores(q, k, grid, block)
    expect = 0.5 * np.outer(alpha, beta) * float(u @ u)   # scale = 1/sqrt(4)
    assert np.allclose(s[0], expect, rtol=1e-14, atol=0)
    sel = oracle.vsa_select(s, 2)
    # positive alpha prefers large beta (blocks 1, 2); negative alpha prefers small beta (0, 3)
    assert sel[0, 0].tolist() == [1, 2] and sel[0, 2].tolist() == [1, 2] and sel[0, 3].tolist() == [1, 2]
    assert sel[0, 1].tolist() == [0, 3]
    assert nblk == 4


def test_select_ties_take_lowest_ids_and_full_k_takes_all():
    s = np.zeros((1, 3, 6))
    assert oracle.vsa_select(s, 4)[0, 0].tolist() == [0, 1, 2, 3]
    s[0, 1] = [1.0, 5.0, 5.0, -2.0, 5.0, 0.0]
    assert oracle.vsa_select(s, 2)[0, 1].tolist() == [1, 2]
    assert oracle.vsa_select(s, 3)[0, 1].tolist() == [1, 2, 4]
    assert oracle.vsa_select(s, 4)[0, 1].tolist() == [0, 1, 2, 4]
    assert oracle.vsa_select(s, 6)[0, 2].tolist() == list(range(6))
    with pytest.raises(ValueError):
        oracle.vsa_select(s, 7)


def test_full_selection_equals_dense_attention():
    grid, block = (3, 5, 6), (2, 2, 4)
    N, H, D = 90, 2, 8
    q, k, v = (_normal(s, (N, H, D)) for s in (2, 3, 4))
    nblk = oracle.vsa_block_count(grid, block)
    sel = np.tile(np.arange(nblk), (H, nblk, 1))
    o, lse = oracle.vsa_attention(q, k, v, grid, block, sel)
    od, lsed = oracle.varlen_attention(q, k, v, [0, N])
    assert np.allclose(o, od, rtol=0, atol=1e-12) and np.allclose(lse, lsed, rtol=0, atol=1e-12)


def test_self_selection_equals_window_attention_with_block_windows():
    grid, block = (5, 9, 11), (4, 4, 4)
    N, H, D = 5 * 9 * 11, 2, 8
    q, k, v = (_normal(s, (N, H, D)) for s in (5, 6, 7))
    nblk = oracle.vsa_block_count(grid, block)
    sel = np.tile(np.arange(nblk)[:, None], (H, 1, 1))          # each block selects itself (k = 1)
    o, lse = oracle.vsa_attention(q, k, v, grid, block, sel)
    perm, cu = oracle.window_partition(grid, block, (0, 0, 0))   # windows = blocks, no shift
    op, lsep = oracle.varlen_attention(oracle.window_pack(q, perm), oracle.window_pack(k, perm),
                                       oracle.window_pack(v, perm), cu)
    assert np.allclose(o, oracle.window_unpack(op, perm), rtol=0, atol=1e-12)
    assert np.allclose(lse, oracle.window_unpack(lsep.T, perm).T, rtol=0, atol=1e-12)


def _bruteforce(q, k, v, blk, sel, scale):
    """Pure-Python masked softmax: key j is visible to query i iff blk[j] is in sel[h][blk[i]]."""
    N, H, D = q.shape
    o = np.zeros((N, H, D))
    lse = np.zeros((H, N))
    for h in range(H):
        for i in range(N):
            keep = set(int(b) for b in sel[h][blk[i]])
            js = [j for j in range(N) if int(blk[j]) in keep]
            sc = [scale * math.fsum(q[i, h, d] * k[j, h, d] for d in range(D)) for j in js]
            mx = max(sc)
            ex = [math.exp(x - mx) for x in sc]
            tot = math.fsum(ex)
            for d in range(D):
                o[i, h, d] = math.fsum(e * v[j, h, d] for e, j in zip(ex, js)) / tot
            lse[h, i] = mx + math.log(tot)
    return o, lse


def test_random_selection_matches_bruteforce_and_ignores_list_order():
    grid, block = (3, 4, 5), (2, 2, 2)
    N, H, D = 60, 2, 4
    q, k, v = (_normal(s, (N, H, D)) for s in (8, 9, 10))
    nblk = oracle.vsa_block_count(grid, block)                   # 2 x 2 x 3 = 12
    rng = np.random.default_rng(11)
    sel = np.stack([np.stack([np.sort(rng.choice(nblk, 3, replace=False)) for _ in range(nblk)])
                    for _ in range(H)])
    o, lse = oracle.vsa_attention(q, k, v, grid, block, sel)
    ob, lseb = _bruteforce(q, k, v, oracle.vsa_block_ids(grid, block), sel, 0.5)
    assert np.allclose(o, ob, rtol=0, atol=1e-12) and np.allclose(lse, lseb, rtol=0, atol=1e-12)
    o2, lse2 = oracle.vsa_attention(q, k, v, grid, block, sel[:, :, ::-1])
    assert np.allclose(o, o2, rtol=0, atol=1e-13) and np.allclose(lse, lse2, rtol=0, atol=1e-13)


def test_selection_from_scores_end_to_end_on_tiny_grid():
    # the selected blocks' keys are the only ones with weight: perturbing any other key block
    # leaves the output unchanged, perturbing a selected one changes it
    grid, block = (4, 4, 8), (2, 2, 2)
    N, H, D = 128, 1, 4
    q, k, v = (_normal(s, (N, H, D)) for s in (12, 13, 14))
    sel = oracle.vsa_select(oracle.vsa_block_scores(q, k, grid, block), 3)
    o, _ = oracle.vsa_attention(q, k, v, grid, block, sel)
    ids = oracle.vsa_block_ids(grid, block)
    a = 5
    rows = np.nonzero(ids == a)[0]
    other = [b for b in range(oracle.vsa_block_count(grid, block)) if b not in sel[0, a]][0]
    k2, v2 = k.copy(), v.copy()
    k2[ids == other] += 10.0
    v2[ids == other] -= 7.0
    o2, _ = oracle.vsa_attention(q, k2, v2, grid, block, sel)
    assert np.array_equal(o[rows], o2[rows])
    v3 = v.copy()
    v3[ids == sel[0, a, 0]] += 1.0
    o3, _ = oracle.vsa_attention(q, k, v3, grid, block, sel)
    assert not np.allclose(o[rows], o3[rows])


def test_row_subset_matches_full():
    grid, block = (3, 5, 6), (2, 2, 4)
    N, H, D = 90, 2, 8
    q, k, v = (_normal(s, (N, H, D)) for s in (15, 16, 17))
    sel = oracle.vsa_select(oracle.vsa_block_scores(q, k, grid, block), 2)
    o, lse = oracle.vsa_attention(q, k, v, grid, block, sel)
    rows = np.array([0, 7, 33, 89])
    os_, lses = oracle.vsa_attention(q, k, v, grid, block, sel, rows=rows)
    # same arithmetic on fewer rows (BLAS may block a smaller product differently: 1e-14)
    assert np.allclose(os_[rows], o[rows], rtol=0, atol=1e-14)
    assert np.allclose(lses[:, rows], lse[:, rows], rtol=0, atol=1e-14)
    assert np.isnan(os_[1]).all()


def test_a_repeated_block_counts_its_keys_twice():
    """Listing a block twice doubles the weight of each of its keys.  With every block of a list
    repeated, numerator and denominator double: the output is unchanged and the LSE grows by
    exactly ln 2.  With one block of [a, b] repeated, the result equals attention over [a, b]
    whose scores on a's keys are raised by ln 2 (a pure-Python masked softmax)."""
    grid, block = (4, 4, 8), (2, 2, 4)   # 2 x 2 x 2 = 8 blocks of 16 tokens
    N, H, D = 128, 1, 4
    q, k, v = (_normal(s, (N, H, D)) for s in (31, 32, 33))
    nblk = oracle.vsa_block_count(grid, block)
    ids = oracle.vsa_block_ids(grid, block)
    once = np.tile(np.array([1, 5]), (H, nblk, 1))
    twice = np.tile(np.array([1, 1, 5, 5]), (H, nblk, 1))
    o1, lse1 = oracle.vsa_attention(q, k, v, grid, block, once)
    o2, lse2 = oracle.vsa_attention(q, k, v, grid, block, twice)
    assert np.allclose(o2, o1, rtol=0, atol=1e-12)
    assert np.allclose(lse2, lse1 + math.log(2.0), rtol=0, atol=1e-12)
    # [1, 1, 5]: block 1's keys weigh double
    o3, lse3 = oracle.vsa_attention(q, k, v, grid, block, np.tile(np.array([1, 1, 5]), (H, nblk, 1)))
    keys = np.concatenate([np.nonzero(ids == 1)[0], np.nonzero(ids == 5)[0]])
    bonus = np.where(ids[keys] == 1, math.log(2.0), 0.0)
    for i in (0, 37, 127):
        s = [sum(q[i, 0, d] * k[j, 0, d] for d in range(D)) / math.sqrt(D) + b for j, b in zip(keys, bonus)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        z = sum(w)
        ref = [sum(wi * v[j, 0, d] for wi, j in zip(w, keys)) / z for d in range(D)]
        assert np.allclose(o3[i, 0], ref, rtol=0, atol=1e-12)
        assert abs(lse3[0, i] - (m + math.log(z))) < 1e-12
