"""Pins of the CPU fp64 oracle against what the pages and the mathematics fix (no GPU).

Each pin is chosen so that a plausible mistake in the oracle fails at least one of them:
  * a leak across segments / a causal mask        -> worked example, perturbation, brute force
  * a dropped or wrong softmax scale, a transposed operand, a wrong sign -> brute force, SDPA
  * wrong rotation pairing / sign                 -> complex-exponential form, quarter turns
  * wrong frequency ladder (exponent, restart per band) -> exact special angles
  * time shift with the wrong ratio or wrong axis -> printed 396.67, closed forms, band isolation
  * window partition off by one / wrong order     -> closed-form counts and sums, brute force
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import (TAG_AUDIO, TAG_TEXT, TAG_VIDEO, random_packed, tiny_example)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------------------------
# cu_seqlens semantics (the pages' worked example)
# ----------------------------------------------------------------------------------------------

def test_worked_example_cu_seqlens_layout(golden_dir):
    g = _load(golden_dir, "cu_seqlens_worked_example.json")
    wl = tiny_example()
    assert list(wl.cu_seqlens) == g["cu_seqlens_three"]
    assert list(np.concatenate([[0], np.cumsum(g["lengths_two"])])) == g["cu_seqlens_two"]
    assert list(np.concatenate([[0], np.cumsum(g["lengths_three"])])) == g["cu_seqlens_three"]


def test_worked_example_zero_weight_outside_segment(golden_dir):
    g = _load(golden_dir, "cu_seqlens_worked_example.json")
    wl = tiny_example()
    i = g["query_row"]
    for h in range(wl.num_heads):
        w = oracle.attention_weights(wl.q, wl.k, wl.cu_seqlens, i, h)
        for lo, hi in g["zero_weight_key_ranges"]:
            assert np.all(w[lo:hi + 1] == 0.0)
        a, b = g["visible_keys_first_last"]
        vis = w[a:b + 1]
        assert np.all(vis > 0.0)  # non-causal: keys after row 15 are weighted too
        assert abs(math.fsum(vis) - 1.0) < 1e-14


def _perturb_outside(t, lo, hi, rng, mode):
    t = t.clone()
    sel = torch.ones(t.shape[0], dtype=torch.bool)
    sel[lo:hi] = False
    if mode == "random":
        t[sel] = torch.from_numpy(rng.standard_normal(size=(int(sel.sum()),) + tuple(t.shape[1:])) * 50).to(t.dtype)
    elif mode == "inf":
        t[sel] = float("inf")
    elif mode == "-inf":
        t[sel] = float("-inf")
    else:
        t[sel] = float("nan")
    return t


@pytest.mark.parametrize("mode", ["random", "inf", "-inf", "nan"])
def test_perturbing_other_segments_and_pad_leaves_segment_unchanged(mode):
    wl = tiny_example(capacity=64)  # 19 NaN pad rows after the 45 valid ones
    cu = wl.cu_seqlens
    o_ref, lse_ref = oracle.varlen_attention(wl.q, wl.k, wl.v, cu)
    rng = np.random.default_rng(7)
    for g in range(wl.num_segments):
        lo, hi = int(cu[g]), int(cu[g + 1])
        q = _perturb_outside(wl.q, lo, hi, rng, mode)
        k = _perturb_outside(wl.k, lo, hi, rng, mode)
        v = _perturb_outside(wl.v, lo, hi, rng, mode)
        o, lse = oracle.varlen_attention(q, k, v, cu)
        assert np.array_equal(o[lo:hi], o_ref[lo:hi])
        assert np.array_equal(lse[:, lo:hi], lse_ref[:, lo:hi])


# ----------------------------------------------------------------------------------------------
# attention math
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("lengths", [[10, 20, 15], [1, 7, 0, 13], [5, 1, 1, 9, 2], [23]])
def test_varlen_equals_dense_masked_bruteforce(lengths):
    wl = random_packed(11 + len(lengths), lengths, heads=2, head_dim=8, capacity=sum(lengths) + 3)
    o, lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    seg = np.full(wl.capacity, -1)
    for g in range(wl.num_segments):
        seg[wl.cu_seqlens[g]:wl.cu_seqlens[g + 1]] = g
    ob, lseb = oracle.dense_masked_attention_bruteforce(wl.q, wl.k, wl.v, seg)
    N = wl.num_tokens
    assert np.max(np.abs(o[:N] - ob[:N])) < 1e-12
    assert np.max(np.abs(lse[:, :N] - lseb[:, :N])) < 1e-12
    assert np.all(np.isnan(o[N:]))  # pad rows are never produced


def test_single_segment_equals_textbook_sdpa():
    wl = random_packed(21, [37], heads=3, head_dim=16)
    o, _ = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    q = wl.q.double().permute(1, 0, 2)
    k = wl.k.double().permute(1, 0, 2)
    v = wl.v.double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v).permute(1, 0, 2).numpy()
    assert np.max(np.abs(o - ref)) < 1e-12


def test_explicit_scale_is_used():
    wl = random_packed(22, [9, 6], heads=1, head_dim=8)
    seg = np.repeat([0, 1], [9, 6])
    o, lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens, scale=0.3)
    ob, lseb = oracle.dense_masked_attention_bruteforce(wl.q, wl.k, wl.v, seg, scale=0.3)
    assert np.max(np.abs(o - ob)) < 1e-12 and np.max(np.abs(lse - lseb)) < 1e-12


def test_length_one_segment_returns_its_value_row_exactly():
    wl = random_packed(23, [4, 1, 6], heads=2, head_dim=8)
    o, lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    assert np.array_equal(o[4], wl.v[4].double().numpy())
    s = (wl.q[4].double() * wl.k[4].double()).sum(-1).numpy() / math.sqrt(8)
    assert np.allclose(lse[:, 4], s, rtol=0, atol=1e-14)


def test_constant_values_give_that_value():
    wl = random_packed(24, [12, 17], heads=2, head_dim=8)
    v = wl.v.clone()
    v[12:29] = v[12]
    o, _ = oracle.varlen_attention(wl.q, wl.k, v, wl.cu_seqlens)
    assert np.max(np.abs(o[12:29] - v[12].double().numpy())) < 1e-14


def test_identical_keys_lse_is_log_n_plus_score():
    wl = random_packed(25, [33], heads=1, head_dim=8)
    k = wl.k.clone()
    k[:] = k[0]
    o, lse = oracle.varlen_attention(wl.q, k, wl.v, wl.cu_seqlens)
    s = (wl.q.double() * k.double()).sum(-1)[:, 0].numpy() / math.sqrt(8)
    assert np.max(np.abs(lse[0] - (s + math.log(33)))) < 1e-12
    assert np.max(np.abs(o[:, 0] - wl.v[:, 0].double().mean(0).numpy())) < 1e-14


def test_row_subset_matches_full():
    wl = random_packed(26, [40, 25], heads=2, head_dim=8)
    o, lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    rows = np.array([0, 7, 39, 40, 64])
    o2, lse2 = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens, rows=rows)
    assert np.array_equal(o2[rows], o[rows])
    assert np.array_equal(lse2[:, rows], lse[:, rows])
    others = np.setdiff1d(np.arange(65), rows)
    assert np.all(np.isnan(o2[others]))


# ----------------------------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------------------------

def _x(seed, n, h, d):
    return np.random.default_rng(seed).standard_normal((n, h, d))


def test_rope_zero_position_is_identity():
    x = _x(1, 6, 2, 64)
    pos = np.zeros((6, 3), np.float32)
    tag = np.array([0, 1, 2, 1, 0, 2], np.uint8)
    assert np.array_equal(oracle.rope_apply(x, pos, tag), x)


def test_rope_preserves_pair_norms():
    x = _x(2, 20, 3, 64)
    wl = tiny_example()
    y = oracle.rope_apply(x[:20], wl.pos[:20], wl.tag[:20])
    n0 = x[:20, :, 0::2] ** 2 + x[:20, :, 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.max(np.abs(n0 - n1)) < 1e-12


def test_rope_matches_complex_exponential_form():
    # RoFormer's complex form: (x_2i + i x_2i+1) * exp(i * phi_i)
    x = _x(3, 5, 2, 32)
    pos = np.zeros((5, 3), np.float32)
    pos[:, 0] = [0, 1, 2.5, 17, 396.6666666666667]
    tag = np.zeros(5, np.uint8)
    y = oracle.rope_apply(x, pos, tag)
    phi = oracle.rope_angles(pos, tag, 32)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * phi)[:, None, :]
    assert np.max(np.abs(y[..., 0::2] - z.real)) < 1e-12
    assert np.max(np.abs(y[..., 1::2] - z.imag)) < 1e-12


def test_rope_exact_special_angles_pin_the_ladder():
    """theta_i = base^(-2i/d): pair 0 turns by t; pair d/4 turns by t/100 at base 10^4."""
    D = 64
    x = np.zeros((2, 1, D))
    x[:, 0, 0::2] = 1.0  # every pair starts at (1, 0)
    pos = np.zeros((2, 3), np.float32)
    pos[0, 0] = np.float32(math.pi)         # pair 0 (theta = 1) turns half way
    pos[1, 0] = np.float32(50.0 * math.pi)  # pair 16 (theta = 10^-2) turns a quarter
    tag = np.array([TAG_TEXT, TAG_AUDIO], np.uint8)
    y = oracle.rope_apply(x, pos, tag)
    t0, t1 = float(pos[0, 0]), float(pos[1, 0])
    assert abs(y[0, 0, 0] - math.cos(t0)) < 1e-15 and abs(y[0, 0, 0] + 1.0) < 1e-12
    assert abs(y[1, 0, 32] - math.cos(t1 / 100.0)) < 1e-12 and abs(y[1, 0, 33] - 1.0) < 1e-9
    # the geometric ratio between neighbouring pairs is base^(-2/D)
    f = oracle.rope_inv_freq(10000.0, D)
    assert f[0] == 1.0 and abs(f[D // 4] - 0.01) < 1e-16
    assert np.max(np.abs(f[1:] / f[:-1] - 10000.0 ** (-2.0 / D))) < 1e-14


def test_video_bands_restart_their_ladders_and_are_isolated():
    D = 64
    dt, dh, dw = oracle.video_axis_split(D)
    assert (dt, dh, dw) == (32, 16, 16)
    x = _x(4, 1, 1, D)
    base = np.zeros((1, 3), np.float32)
    tag = np.array([TAG_VIDEO], np.uint8)
    y0 = oracle.rope_apply(x, base, tag)
    for axis, (lo, hi) in enumerate([(0, dt), (dt, dt + dh), (dt + dh, D)]):
        p = base.copy()
        p[0, axis] = np.float32(math.pi)
        y = oracle.rope_apply(x, p, tag)
        changed = np.nonzero(np.abs(y - y0)[0, 0] > 1e-12)[0]
        assert changed.min() >= lo and changed.max() < hi
        # the first pair of each band has theta = 1: a half turn negates it exactly
        # (float32(pi) is within 1e-7 of pi; a ladder that did not restart would turn by 0.03 rad)
        assert abs(y[0, 0, lo] + x[0, 0, lo]) < 1e-6 and abs(y[0, 0, lo + 1] + x[0, 0, lo + 1]) < 1e-6


def test_rope_relative_position_invariance_within_modality():
    wl = tiny_example()
    rng = np.random.default_rng(5)
    q = rng.standard_normal((45, 2, 64))
    k = rng.standard_normal((45, 2, 64))
    ref_q = oracle.rope_apply(q, wl.pos, wl.tag)
    ref_k = oracle.rope_apply(k, wl.pos, wl.tag)
    dots = np.einsum("ihd,jhd->hij", ref_q, ref_k)
    for tg, axes in [(TAG_TEXT, [0]), (TAG_AUDIO, [0]), (TAG_VIDEO, [0, 1, 2])]:
        for ax in axes:
            pos = wl.pos.astype(np.float64).copy()
            pos[wl.tag == tg, ax] += 123.25
            rq = oracle.rope_apply(q, pos, wl.tag)
            rk = oracle.rope_apply(k, pos, wl.tag)
            d2 = np.einsum("ihd,jhd->hij", rq, rk)
            sel = np.nonzero(wl.tag == tg)[0]
            blk = np.ix_(range(2), sel, sel)
            assert np.max(np.abs(d2[blk] - dots[blk])) < 1e-10
            # and the same shift does change dot products against the other modalities
            other = np.nonzero(wl.tag != tg)[0]
            assert np.max(np.abs(d2[np.ix_(range(2), sel, other)] - dots[np.ix_(range(2), sel, other)])) > 1e-3


def test_rotation_composition_closed_form():
    # R(a)^T R(b) = R(b - a) per pair: rotating q by a and k by b gives q . R(b-a) k
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((1, 1, 16))
    pa = np.array([[3.0, 0, 0]])
    pb = np.array([[10.5, 0, 0]])
    tag = np.array([TAG_TEXT], np.uint8)
    lhs = np.sum(oracle.rope_apply(q, pa, tag) * oracle.rope_apply(k, pb, tag))
    rhs = np.sum(q * oracle.rope_apply(k, pb - pa, tag))
    assert abs(lhs - rhs) < 1e-12


# ----------------------------------------------------------------------------------------------
# continuation time shift
# ----------------------------------------------------------------------------------------------

def test_time_shift_printed_example(golden_dir):
    g = _load(golden_dir, "continuation_time_shift.json")
    s = oracle.continuation_time_shift(g["start_frame"], g["audio_hz"], g["video_fps"])
    assert round(s, g["printed_decimals"]) == g["printed_offset"]
    assert s == float(Fraction(g["start_frame"] * g["audio_hz"], g["video_fps"]))
    assert s != round(s)  # decimals are kept


def test_time_shift_set_closed_forms():
    vals = [oracle.continuation_time_shift(s) for s in (0, 119, 238, 357)]
    assert vals[0] == 0.0 and vals[3] == 595.0
    assert vals[1] == float(Fraction(595, 3)) and vals[2] == float(Fraction(1190, 3))


def test_time_shift_moves_only_time_band_and_only_its_request():
    D = 64
    rng = np.random.default_rng(8)
    x = rng.standard_normal((6, 1, D))
    pos = np.array([[1, 0, 0], [2, 1, 3], [0, 0, 0], [1, 0, 0], [2, 1, 3], [0, 0, 0]], np.float32)
    tag = np.array([TAG_TEXT, TAG_VIDEO, TAG_AUDIO] * 2, np.uint8)
    cu_req = [0, 3, 6]
    y0 = oracle.rope_apply(x, pos, tag, cu_req, [0.0, 0.0])
    y1 = oracle.rope_apply(x, pos, tag, cu_req, [0.0, 238.0])
    assert np.array_equal(y0[:3], y1[:3])             # request 0 not shifted
    assert np.array_equal(y0[4, :, 32:], y1[4, :, 32:])  # video h/w bands untouched
    assert np.max(np.abs(y0[4, :, :32] - y1[4, :, :32])) > 1e-3
    # shifting request 1 by s equals placing its tokens at t + s*40/24 (decimals kept)
    p2 = pos.astype(np.float64).copy()
    p2[3:, 0] += 238 * 40 / 24
    y2 = oracle.rope_apply(x, p2, tag)
    assert np.max(np.abs(y2[3:] - y1[3:])) < 1e-12


def test_uniform_request_shift_leaves_attention_unchanged():
    wl = tiny_example()
    qa = oracle.rope_apply(wl.q, wl.pos, wl.tag, [0, 45], [0.0])
    ka = oracle.rope_apply(wl.k, wl.pos, wl.tag, [0, 45], [0.0])
    qb = oracle.rope_apply(wl.q, wl.pos, wl.tag, [0, 45], [238.0])
    kb = oracle.rope_apply(wl.k, wl.pos, wl.tag, [0, 45], [238.0])
    assert np.max(np.abs(qa - qb)) > 1e-2  # the rotation itself does change
    oa, la = oracle.varlen_attention(qa, ka, wl.v, wl.cu_seqlens)
    ob, lb = oracle.varlen_attention(qb, kb, wl.v, wl.cu_seqlens)
    assert np.max(np.abs(oa - ob)) < 1e-11 and np.max(np.abs(la - lb)) < 1e-11


# ----------------------------------------------------------------------------------------------
# window partition
# ----------------------------------------------------------------------------------------------

GRID5, WIN5, SH5 = (32, 48, 84), (4, 8, 8), (2, 4, 4)


def test_window_counts_closed_form():
    assert oracle.window_count(GRID5, WIN5, (0, 0, 0)) == 8 * 6 * 11 == 528
    assert oracle.window_count(GRID5, WIN5, SH5) == 9 * 7 * 11 == 693


@pytest.mark.parametrize("shift,sum_sq", [((0, 0, 0), 128 * 384 * 656), (SH5, 120 * 352 * 656)])
def test_window_sizes_closed_form(shift, sum_sq):
    perm, cu = oracle.window_partition(GRID5, WIN5, shift)
    n = np.diff(cu).astype(np.int64)
    assert cu[0] == 0 and cu[-1] == 32 * 48 * 84 == 129024
    assert np.all(n > 0)
    assert int(np.sum(n * n)) == sum_sq
    assert np.array_equal(np.sort(perm), np.arange(129024))  # bijection


def _bruteforce_partition(grid, win, shift):
    T, H, W = grid
    out_perm, out_cu = [], [0]
    ranges = []
    for a, (L, w, s) in enumerate(zip(grid, win, shift)):
        r = []
        i = 0
        while True:
            lo, hi = max(0, i * w - s), min(L, (i + 1) * w - s)
            if lo >= L:
                break
            r.append((lo, hi))
            i += 1
        ranges.append(r)
    for (t0, t1) in ranges[0]:
        for (h0, h1) in ranges[1]:
            for (w0, w1) in ranges[2]:
                for t in range(t0, t1):
                    for h in range(h0, h1):
                        for w in range(w0, w1):
                            out_perm.append(t * H * W + h * W + w)
                out_cu.append(len(out_perm))
    return np.array(out_perm), np.array(out_cu)


@pytest.mark.parametrize("grid,win,shift", [((5, 6, 7), (2, 4, 4), (1, 2, 2)), ((4, 8, 9), (4, 8, 8), (0, 0, 0)),
                                            ((3, 5, 11), (2, 2, 4), (1, 1, 2)), ((1, 1, 1), (4, 8, 8), (2, 4, 4))])
def test_window_partition_matches_bruteforce(grid, win, shift):
    perm, cu = oracle.window_partition(grid, win, shift)
    bp, bc = _bruteforce_partition(grid, win, shift)
    assert np.array_equal(perm, bp) and np.array_equal(cu, bc)
    # each token's window recomputed independently by floor((x+s)/w)
    ids = oracle.window_ids(grid, win, shift)
    T, H, W = grid
    for x in range(T * H * W):
        t, h, w = x // (H * W), (x // W) % H, x % W
        key = ((t + shift[0]) // win[0], (h + shift[1]) // win[1], (w + shift[2]) // win[2])
        n_h = -(-(H + shift[1]) // win[1])
        n_w = -(-(W + shift[2]) // win[2])
        assert ids[x] == (key[0] * n_h + key[1]) * n_w + key[2]


def test_pack_unpack_roundtrip_is_identity():
    grid = (3, 5, 11)
    perm, _ = oracle.window_partition(grid, (2, 2, 4), (1, 1, 2))
    x = torch.randn(3 * 5 * 11, 2, 8).to(torch.bfloat16)
    assert torch.equal(oracle.window_unpack(oracle.window_pack(x, perm), perm), x)


def test_window_attention_equals_masked_attention_in_original_order():
    grid, win, shift = (2, 4, 6), (2, 4, 4), (1, 2, 2)
    n = 48
    rng = np.random.default_rng(9)
    q, k, v = (torch.from_numpy(rng.standard_normal((n, 1, 8)).astype(np.float32)).to(torch.bfloat16)
               for _ in range(3))
    perm, cu = oracle.window_partition(grid, win, shift)
    o_packed, _ = oracle.varlen_attention(oracle.window_pack(q, perm), oracle.window_pack(k, perm),
                                          oracle.window_pack(v, perm), cu)
    o = oracle.window_unpack(o_packed, perm)
    ob, _ = oracle.dense_masked_attention_bruteforce(q, k, v, oracle.window_ids(grid, win, shift))
    assert np.max(np.abs(o - ob)) < 1e-12


def test_trim_padding_numbers(golden_dir):
    g = _load(golden_dir, "trim_padding.json")
    assert g["aligned_tokens"] - g["valid_tokens"] == g["padding_tokens"]
    assert 558 + 200 + 29 * 40 * 50 == g["valid_tokens"]
    assert -(-g["valid_tokens"] // 64) * 64 == g["aligned_tokens"]


def test_rope_row_subset_matches_full():
    wl = tiny_example()
    full = oracle.rope_apply(wl.q, wl.pos, wl.tag, [0, 20, 45], [0.0, 119.0])
    rows = np.array([3, 15, 19, 20, 44])
    sub = oracle.rope_apply(wl.q, wl.pos, wl.tag, [0, 20, 45], [0.0, 119.0], rows=rows)
    assert np.array_equal(sub, full[rows])


# ----------------------------------------------------------------------------------------------
# non-default RoPE configuration: a base per modality, an uneven video band split, other rates
# in the continuation shift ([H3-vLLM] §3: the tag selects the frequencies)
# ----------------------------------------------------------------------------------------------

# bases whose square roots are whole numbers, so a quarter turn of the pair at index d/4 of a
# band (theta = base^(-1/2)) falls at a coordinate that is a simple multiple of pi
CUSTOM_BASES = dict(base_text=2500.0, base_video=900.0, base_audio=400.0)  # sqrt 50, 30, 20
CUSTOM_SPLIT = (24, 64, 40)  # three different widths at D = 128: t, h, w


def _custom_cfg(**kw):
    return oracle.RopeConfig(**CUSTOM_BASES, video_dims_t=CUSTOM_SPLIT[0], video_dims_h=CUSTOM_SPLIT[1],
                             video_dims_w=CUSTOM_SPLIT[2], **kw)


def _unit_pairs(n, D):
    x = np.zeros((n, 1, D))
    x[:, 0, 0::2] = 1.0  # every pair starts at (1, 0)
    return x


def test_custom_bases_quarter_turn_at_a_quarter_of_each_ladder():
    """Pair D/4 of a text / audio row turns by t * base^(-1/2): a quarter turn at t = sqrt(base) pi/2.
    With distinct bases a swapped base_text / base_audio (or video) turns by another angle."""
    D = 128
    cfg = _custom_cfg()
    x = _unit_pairs(3, D)
    pos = np.zeros((3, 3), np.float64)
    pos[0, 0] = 25.0 * math.pi   # text:  sqrt(2500) = 50 -> 25 pi / 50 = pi / 2
    pos[1, 0] = 10.0 * math.pi   # audio: sqrt(400)  = 20 -> 10 pi / 20 = pi / 2
    pos[2, 0] = 6.0 * math.pi    # video time band (24 dims): pair 6 turns by 6 pi / 30 ... see below
    tag = np.array([TAG_TEXT, TAG_AUDIO, TAG_VIDEO], np.uint8)
    y = oracle.rope_apply(x, pos, tag, cfg=cfg)
    for r in (0, 1):  # pair D/4 = 32 -> dims 64, 65 at (0, 1)
        assert abs(y[r, 0, 64]) < 1e-12 and abs(y[r, 0, 65] - 1.0) < 1e-12, r
    # video time band of width 24: its pair 24/4 = 6 (dims 12, 13) has theta = 900^(-1/2) = 1/30,
    # so t = 6 pi turns it by pi / 5; its pair 0 (theta = 1) turns by 6 pi = a whole number of turns
    assert abs(y[2, 0, 12] - math.cos(math.pi / 5)) < 1e-12 and abs(y[2, 0, 13] - math.sin(math.pi / 5)) < 1e-12
    assert abs(y[2, 0, 0] - 1.0) < 1e-12 and abs(y[2, 0, 1]) < 1e-12
    # the pair just before a band's quarter point is not at the special angle (the ladder is
    # anchored per band, not per head)
    assert abs(y[0, 0, 62]) > 1e-3


def test_custom_video_split_bands_move_only_their_dims_and_restart():
    """Split 24 / 64 / 40: moving t, h or w changes exactly dims [0,24), [24,88), [88,128), the
    first pair of each band (theta = 1) is negated by a half turn, and the pair at a quarter of
    each band turns by coordinate * 900^(-1/2)."""
    D = 128
    cfg = _custom_cfg()
    dt, dh, dw = oracle.video_axis_split(D, *CUSTOM_SPLIT)
    assert (dt, dh, dw) == CUSTOM_SPLIT
    bands = [(0, dt), (dt, dt + dh), (dt + dh, D)]
    x = np.random.default_rng(11).standard_normal((1, 1, D))
    tag = np.array([TAG_VIDEO], np.uint8)
    y0 = oracle.rope_apply(x, np.zeros((1, 3)), tag, cfg=cfg)
    assert np.array_equal(y0, x)
    for axis, (lo, hi) in enumerate(bands):
        p = np.zeros((1, 3))
        p[0, axis] = math.pi
        y = oracle.rope_apply(x, p, tag, cfg=cfg)
        changed = np.nonzero(np.abs(y - x)[0, 0] > 1e-12)[0]
        assert changed.min() == lo and changed.max() == hi - 1, axis
        assert abs(y[0, 0, lo] + x[0, 0, lo]) < 1e-12 and abs(y[0, 0, lo + 1] + x[0, 0, lo + 1]) < 1e-12
        # quarter turn of the band's pair (hi - lo) / 4 at coordinate 15 pi (15 pi / 30 = pi / 2)
        u = _unit_pairs(1, D)
        p[0, axis] = 15.0 * math.pi
        yu = oracle.rope_apply(u, p, tag, cfg=cfg)
        k = lo + 2 * ((hi - lo) // 4)
        assert abs(yu[0, 0, k]) < 1e-12 and abs(yu[0, 0, k + 1] - 1.0) < 1e-12, axis


def test_custom_shift_rates_closed_form():
    """s * audio_hz / video_fps with other rates: 330 * 48 / 25 = 633.6, and a start frame of
    25 pi / 48 at 48 / 25 moves t by exactly pi (pair 0 of a text row at t = 0 is negated); with
    the rates swapped it would move by 25^2 pi / 48^2."""
    cfg = _custom_cfg(audio_hz=48.0, video_fps=25.0)
    assert oracle.continuation_time_shift(330.0, cfg.audio_hz, cfg.video_fps) == float(Fraction(330 * 48, 25))
    off = oracle.rope.request_time_offsets(4, [0, 2, 4], [0.0, 330.0], cfg)
    assert np.array_equal(off, [0.0, 0.0, float(Fraction(330 * 48, 25)), float(Fraction(330 * 48, 25))])
    x = _unit_pairs(2, 128)
    pos = np.zeros((2, 3))
    tag = np.array([TAG_TEXT, TAG_TEXT], np.uint8)
    y = oracle.rope_apply(x, pos, tag, [0, 1, 2], [0.0, 25.0 * math.pi / 48.0], cfg=cfg)
    assert np.array_equal(y[0], x[0])                     # request 0: no shift
    assert abs(y[1, 0, 0] + 1.0) < 1e-12 and abs(y[1, 0, 1]) < 1e-12
