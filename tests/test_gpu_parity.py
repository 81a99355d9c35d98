"""GPU parity of the CUDA path (through the C ABI) against the CPU fp64 oracle.

Tolerances (bf16 storage, fp32 math):
  * bf16 outputs (RoPE, attention): max |err| <= 2e-2 and mean |err| <= 2e-3 against fp64;
  * LSE: |err| <= 1e-4 * max(|lse|, 1)  (relative, with a floor of 1 for near-zero values);
  * integer outputs (perm, cu_seqlens) and pure copies (window gather / restore): bit-exact.
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


def _close(got, ref, what, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs and err.mean() <= mean_abs, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"
    return err.max(), err.mean()


def _lse_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)
    assert rel.max() <= LSE_REL, f"{what}: lse rel {rel.max():.3e}"


def _to(dev, wl):
    return dict(q=wl.q.to(dev), k=wl.k.to(dev), v=wl.v.to(dev), pos=torch.from_numpy(wl.pos).to(dev),
                tag=torch.from_numpy(wl.tag).to(dev), cu=torch.from_numpy(wl.cu_seqlens).to(dev),
                cu_req=torch.from_numpy(wl.cu_requests).to(dev),
                frames=torch.from_numpy(wl.start_frames).to(dev))


def _sample_rows(cu, seed, edge=128, frac=64):
    """Every row of short segments, the first/last `edge` rows of each segment, 1/frac of the rest."""
    rng = np.random.default_rng(seed)
    rows = []
    for g in range(len(cu) - 1):
        a, b = int(cu[g]), int(cu[g + 1])
        if b - a <= 3 * edge:
            rows.append(np.arange(a, b))
            continue
        rows += [np.arange(a, a + edge), np.arange(b - edge, b)]
        mid = np.arange(a + edge, b - edge)
        rows.append(rng.choice(mid, size=max(1, mid.size // frac), replace=False))
    return np.unique(np.concatenate(rows))


def _run_rope(h3, d, wl):
    qr, kr = torch.empty_like(d["q"]), torch.empty_like(d["k"])
    h3.rope_apply(d["q"], d["k"], d["pos"], d["tag"], d["cu_req"], d["frames"], num_tokens=wl.num_tokens,
                  q_out=qr, k_out=kr)
    return qr, kr


PACKED = {
    "tiny_example": lambda: W.tiny_example(capacity=64),
    "single_request_4k": lambda: W.single_request_4k(capacity=4160),
    "continuation_batch": lambda: W.continuation_batch(),
    "continuation_batch_4seg": lambda: W.continuation_batch(per_request_segments=True),
    "h3_full_request": lambda: W.h3_full_request(),
}
FULL_CHECK = {"tiny_example", "single_request_4k"}


@pytest.fixture(scope="module", params=list(PACKED))
def packed_case(request, h3, dev):
    wl = PACKED[request.param]()
    d = _to(dev, wl)
    qr, kr = _run_rope(h3, d, wl)
    o, lse = h3.varlen_attn_fwd(qr, kr, d["v"], d["cu"], wl.max_seqlen, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    full = request.param in FULL_CHECK
    rows = np.arange(wl.num_tokens) if full else _sample_rows(wl.cu_seqlens, seed=len(request.param))
    res = dict(wl=wl, rows=rows, full=full, q_rot=qr.cpu(), k_rot=kr.cpu(), o=o.cpu(), lse=lse.cpu())
    del d, qr, kr, o, lse
    torch.cuda.empty_cache()
    return request.param, res


def test_rope_parity(packed_case):
    name, r = packed_case
    wl, rows = r["wl"], r["rows"]
    for t_in, t_out in ((wl.q, r["q_rot"]), (wl.k, r["k_rot"])):
        ref = oracle.rope_apply(t_in, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, rows=rows)
        _close(t_out[rows].float().numpy(), ref, f"{name} rope")


@pytest.mark.parametrize("D,dims", [(128, (32, 48, 48)), (64, (16, 24, 24))])
def test_rope_custom_config_against_oracle(h3, dev, D, dims):
    """Non-default RoPE settings: a base per modality, a video band split other than D/2:D/4:D/4
    and other sample rates in the continuation shift (s * audio_hz / video_fps), with two
    requests whose start frames differ."""
    wl = W.random_packed(41 + D, [60, 200, 90, 150], heads=2, head_dim=D, capacity=520)
    N = wl.num_tokens
    cu_req = np.array([0, 260, N], np.int32)
    frames = np.array([17.0, 330.0], np.float32)
    cfg_h = h3.RopeConfig(base_text=5000.0, base_video=20000.0, base_audio=1000.0,
                          video_dims_t=dims[0], video_dims_h=dims[1], video_dims_w=dims[2],
                          audio_hz=48.0, video_fps=25.0)
    cfg_o = oracle.RopeConfig(base_text=5000.0, base_video=20000.0, base_audio=1000.0,
                              video_dims_t=dims[0], video_dims_h=dims[1], video_dims_w=dims[2],
                              audio_hz=48.0, video_fps=25.0)
    d = _to(dev, wl)
    qo, ko = h3.rope_apply(d["q"], d["k"], d["pos"], d["tag"], torch.from_numpy(cu_req).to(dev),
                           torch.from_numpy(frames).to(dev), num_tokens=N,
                           q_out=torch.empty_like(d["q"]), k_out=torch.empty_like(d["k"]), cfg=cfg_h)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    for got, src in ((qo, wl.q), (ko, wl.k)):
        ref = oracle.rope_apply(src, wl.pos, wl.tag, cu_req, frames, cfg=cfg_o, num_tokens=N)
        _close(got[:N].float().cpu().numpy(), ref[:N], f"rope custom config D {D}")


def test_attention_parity_on_gpu_rope_output(packed_case):
    """Parity (i): attention alone, the oracle fed the GPU's own bf16 RoPE outputs."""
    name, r = packed_case
    wl, rows = r["wl"], r["rows"]
    ref_o, ref_lse = oracle.varlen_attention(r["q_rot"], r["k_rot"], wl.v, wl.cu_seqlens, rows=rows)
    _close(r["o"][rows].float().numpy(), ref_o[rows], f"{name} attention")
    _lse_close(r["lse"][:, rows].numpy(), ref_lse[:, rows], f"{name} attention")


def test_end_to_end_parity_from_raw_qk(packed_case):
    """Parity (iii): the oracle does its own fp64 RoPE (with the time shift) from raw Q/K.  Short
    segments are checked in full; long ones (sampled cases) on their sampled query rows, against
    every key of the segment."""
    name, r = packed_case
    wl = r["wl"]
    for g in range(wl.num_segments):
        a, b = int(wl.cu_seqlens[g]), int(wl.cu_seqlens[g + 1])
        if b <= a:
            continue
        idx = np.arange(a, b)
        if r["full"] or b - a <= 4096:
            local = np.arange(b - a)
        else:
            local = r["rows"][(r["rows"] >= a) & (r["rows"] < b)] - a
        qo = oracle.rope_apply(wl.q, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, rows=idx)
        ko = oracle.rope_apply(wl.k, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, rows=idx)
        vo = wl.v[a:b].double().numpy()
        ref_o, ref_lse = oracle.varlen_attention(qo, ko, vo, [0, b - a], rows=local)
        _close(r["o"][a:b].float().numpy()[local], ref_o[local], f"{name} e2e seg {g}")
        # The GPU rounds the rotated Q/K to bf16 (storage) before attention.  Since
        # |d lse_i / d S_ij| = P_ij, |lse error| <= max_j |S_ij error| <=
        # scale * 2^-8 * max_j sum_d |q_id||k_jd| (two roundings of at most 2^-9 each).
        scale = 1.0 / np.sqrt(wl.head_dim)
        aq, ak = np.abs(qo[local]).transpose(1, 0, 2), np.abs(ko).transpose(1, 0, 2)  # [H, n, D]
        bound = scale * 2.0 ** -8 * np.matmul(aq, ak.transpose(0, 2, 1)).max(axis=2)
        got = r["lse"][:, a:b].numpy().astype(np.float64)[:, local]
        ref = ref_lse[:, local]
        assert np.all(np.abs(got - ref) <= bound + LSE_REL * np.maximum(np.abs(ref), 1.0)), \
            f"{name} e2e seg {g}: lse outside the bf16-rounding bound"


def test_pad_rows_of_output_untouched(h3, dev):
    wl = W.tiny_example(capacity=64)
    d = _to(dev, wl)
    o = torch.full_like(d["q"], 7.0)
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], 20, out=o)
    torch.cuda.synchronize()
    assert torch.all(o[45:] == 7.0)
    assert torch.all(torch.isfinite(o[:45].float()))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [[1, 127, 128, 129, 0, 255, 256, 257, 2, 383],
                                     [1000, 1, 1, 513], [0, 0, 77], [128 * 5],
                                     # the grid switches from one CTA per SM (max_seqlen <= 2048)
                                     # to one CTA per item just above it
                                     [2048, 5, 0], [2049, 300, 1],
                                     # more segments than the plan orders longest-first (256)
                                     [int(x) for x in np.random.default_rng(23).integers(0, 40, 300)]])
def test_edge_lengths_against_oracle(h3, dev, D, lengths):
    wl = W.random_packed(100 + sum(lengths) % 97, lengths, heads=3, head_dim=D,
                         capacity=sum(lengths) + 61)
    d = _to(dev, wl)
    o = torch.full_like(d["q"], 3.0)
    lse = torch.full((3, wl.capacity), 5.0, device=dev)
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], max(1, wl.max_seqlen), out=o, lse=lse)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    N = wl.num_tokens
    ref_o, ref_lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    if N:
        _close(o[:N].float().cpu().numpy(), ref_o[:N], f"lengths {lengths} D {D}")
        _lse_close(lse[:, :N].cpu().numpy(), ref_lse[:, :N], f"lengths {lengths} D {D}")
    assert torch.all(o[N:] == 3.0) and torch.all(lse[:, N:] == 5.0)


def _random_layout(seed):
    """A seeded random job: 1-47 segments whose lengths mix empty and tiny ones, lengths at and
    around multiples of the 128-row tile, and long ones up to 4,000 rows; 1-8 heads."""
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 48))
    lengths = []
    for _ in range(S):
        kind = rng.random()
        if kind < 0.35:
            lengths.append(int(rng.integers(0, 41)))
        elif kind < 0.7:
            lengths.append(max(0, 128 * int(rng.integers(1, 12)) + int(rng.integers(-2, 3))))
        else:
            lengths.append(int(rng.integers(41, 4001)))
    while sum(lengths) > 14000:
        lengths[int(np.argmax(lengths))] //= 2
    heads = int(rng.choice([1, 2, 3, 5, 8]))
    return lengths, heads, int(rng.integers(0, 200))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("seed", range(8))
def test_random_layouts_against_oracle(h3, dev, D, seed):
    """Seeded random segment layouts through the library's default workspace (which splits the
    last wave when it can): every valid row and its LSE against the oracle, pad rows untouched,
    and the same bytes from a second call."""
    lengths, heads, pad = _random_layout(1000 + seed)
    wl = W.random_packed(1100 + seed + D, lengths, heads=heads, head_dim=D, capacity=sum(lengths) + pad + 1)
    d = _to(dev, wl)
    outs = []
    for _ in range(2):
        o = torch.full_like(d["q"], 3.0)
        lse = torch.full((heads, wl.capacity), 5.0, device=dev)
        h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], max(1, wl.max_seqlen), out=o, lse=lse)
        torch.cuda.synchronize()
        assert h3.get_device_error(dev) == 0
        outs.append((o, lse))
    (o, lse), (o2, lse2) = outs
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    N = wl.num_tokens
    what = f"seed {seed} D {D}: {len(lengths)} segments, max {max(lengths)}, {heads} heads"
    if N:
        ref_o, ref_lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
        _close(o[:N].float().cpu().numpy(), ref_o[:N], what)
        _lse_close(lse[:, :N].cpu().numpy(), ref_lse[:, :N], what)
    assert torch.all(o[N:] == 3.0) and torch.all(lse[:, N:] == 5.0), what


def test_maximum_segment_count_against_oracle(h3, dev):
    """65,535 segments (the most the call accepts) of 0 to 4 rows each: the plan lists far more
    segments than it orders longest-first, most items hold a single short query tile, and the
    empty segments produce nothing."""
    lengths = [int(x) for x in np.random.default_rng(29).integers(0, 5, 65535)]
    wl = W.random_packed(29, lengths, heads=1, head_dim=64, capacity=sum(lengths) + 7)
    d = _to(dev, wl)
    o = torch.full_like(d["q"], 3.0)
    lse = torch.full((1, wl.capacity), 5.0, device=dev)
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], max(1, wl.max_seqlen), out=o, lse=lse)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    N = wl.num_tokens
    ref_o, ref_lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens)
    _close(o[:N].float().cpu().numpy(), ref_o[:N], "65,535 segments")
    _lse_close(lse[:, :N].cpu().numpy(), ref_lse[:, :N], "65,535 segments")
    assert torch.all(o[N:] == 3.0) and torch.all(lse[:, N:] == 5.0)


def _split_entries(h3, ws, S, H, D):
    """(whole items before the last wave, entries of the wave, per-entry chunk field) read back
    from a workspace after a call: the plan header and the split area's entry table."""
    plan = h3.varlen_attn_workspace_size(S, H, 1, D)
    words = ws[:plan].view(torch.int32).cpu().numpy()
    n = int(words[3])
    table = ws[plan:plan + 320 * 32].view(torch.int32).cpu().numpy().reshape(320, 8)
    return int(words[2]), n, table[:n, 7]


def _expected_split_plan(cu, H, sms):
    """The plan's split of the last wave, restated on the host: segments longest first (ties by
    position), items head-major per segment, whole items [0, tail) with tail a multiple of the SM
    count, then the last wave's entries (seg_start, seg_len, head, q0, kv0, kv1, group, split):
    each of its L long items (>= 8 key tiles) cut into min(8, SMs // L, key tiles // 4) chunks."""
    lens = np.diff(np.asarray(cu, np.int64))
    order = sorted(range(len(lens)), key=lambda g: (-lens[g], g))
    items = []
    for g in order:
        pairs = -(-int(lens[g]) // 256)
        for h in range(H):
            for p in range(pairs):
                items.append((int(cu[g]), int(lens[g]), h, int(cu[g]) + 256 * p))
    T = len(items)
    tail = T // sms * sms
    R = T - tail
    if R == 0 or R > 320:
        return tail if R == 0 else T, []
    wave = items[tail:]
    nkv = [-(-ln // 128) for (_, ln, _, _) in wave]
    L = sum(1 for x in nkv if x >= 8)
    c_all = min(8, sms // L) if L else 1
    cs = [max(1, min(c_all, x // 4)) if x >= 8 else 1 for x in nkv]
    if sum(cs) > 320:
        cs = [1] * R
    entries, first = [], 0
    for (a, ln, h, q0), x, c in zip(wave, nkv, cs):
        for ch in range(c):
            entries.append((a, ln, h, q0, x * ch // c, x * (ch + 1) // c, first,
                            (ch << 16 | c) if c > 1 else 0))
        first += c
    return tail, entries


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths,heads", [([8192], 2),            # fewer items than SMs: all split
                                           ([3000, 40, 2500], 3),
                                           ([1024] * 5 + [5000, 1], 1),
                                           ([2000, 700], 8),       # one CTA per SM, looping
                                           ([3520, 256, 320], 24),  # the 4,096-token request's shape
                                           ([1100] * 31 + [40], 1),  # 32 segments: the wave crosses two
                                           ([1100] * 40, 1)])        # more: planned by the plan kernel
def test_split_last_wave_against_oracle_and_whole_items(h3, dev, D, lengths, heads):
    """Long items of the last, partly filled wave are cut into chunks of their key range and
    merged (a workspace with the split area) -- against the oracle, against the same call with a
    plan-only workspace (whole items), and bit-identical call after call (fixed merge order)."""
    wl = W.random_packed(200 + len(lengths) + heads + D, lengths, heads=heads, head_dim=D,
                         capacity=sum(lengths) + 40)
    d = _to(dev, wl)
    S, N = wl.num_segments, wl.num_tokens
    full = torch.empty(h3.varlen_attn_workspace_size(S, heads, wl.max_seqlen, D), dtype=torch.uint8, device=dev)
    plan = torch.empty(h3.varlen_attn_workspace_size(S, heads, 1, D), dtype=torch.uint8, device=dev)
    outs = []
    for ws in (full, full, plan):
        o = torch.full_like(d["q"], 3.0)
        lse = torch.full((heads, wl.capacity), 5.0, device=dev)
        h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], wl.max_seqlen, out=o, lse=lse, workspace=ws)
        torch.cuda.synchronize()
        assert h3.get_device_error(dev) == 0
        outs.append((o, lse))
        if ws is full:
            tail, n, split = _split_entries(h3, full, S, heads, D)
            assert n > 0 and np.any(split != 0), "the last wave was expected to split"
            # the entry table, integer for integer, against the rule restated on the host
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            exp_tail, exp_entries = _expected_split_plan(wl.cu_seqlens, heads, sms)
            plan_bytes = h3.varlen_attn_workspace_size(S, heads, 1, D)
            table = full[plan_bytes:plan_bytes + 320 * 32].view(torch.int32).cpu().numpy().reshape(320, 8)
            assert tail == exp_tail and n == len(exp_entries)
            # the order and item-prefix words: longest first, ties by position
            words = full[:plan_bytes].view(torch.int32).cpu().numpy()
            lens = np.diff(wl.cu_seqlens.astype(np.int64))
            order = sorted(range(S), key=lambda g: (-lens[g], g))
            items = [-(-int(lens[g]) // 256) * heads for g in order]
            assert words[4:4 + S].tolist() == order
            assert words[4 + S:5 + 2 * S].tolist() == [0] + np.cumsum(items).tolist()
            assert np.array_equal(table[:n], np.asarray(exp_entries, np.int32).reshape(-1, 8))
    (o1, l1), (o2, l2), (ow, lw) = outs
    assert torch.equal(o1, o2) and torch.equal(l1, l2)  # deterministic merge
    o_nolse = torch.full_like(d["q"], 3.0)  # the merge without an LSE output writes the same rows
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], wl.max_seqlen, out=o_nolse, workspace=full)
    torch.cuda.synchronize()
    assert torch.equal(o_nolse, o1)
    assert torch.all(o1[N:] == 3.0) and torch.all(l1[:, N:] == 5.0)
    rows = _sample_rows(wl.cu_seqlens, seed=D + heads)
    ref_o, ref_lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens, rows=rows)
    for o, lse, what in ((o1, l1, "split"), (ow, lw, "whole")):
        _close(o[rows].float().cpu().numpy(), ref_o[rows], f"{what} {lengths} x {heads} D {D}")
        _lse_close(lse[:, rows].cpu().numpy(), ref_lse[:, rows], f"{what} {lengths} x {heads} D {D}")
    _close(o1[:N].float().cpu().numpy(), ow[:N].float().cpu().numpy(), f"split vs whole {lengths}")


def test_explicit_softmax_scale(h3, dev):
    wl = W.random_packed(7, [300, 45], heads=2, head_dim=128)
    d = _to(dev, wl)
    o, lse = h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], 300, return_lse=True, softmax_scale=0.05)
    ref_o, ref_lse = oracle.varlen_attention(wl.q, wl.k, wl.v, wl.cu_seqlens, scale=0.05)
    _close(o.float().cpu().numpy(), ref_o, "scale 0.05")
    _lse_close(lse.cpu().numpy(), ref_lse, "scale 0.05")


@pytest.mark.parametrize("fill", [float("nan"), float("inf"), -float("inf"), 1e4])
def test_out_of_segment_rows_cannot_leak(h3, dev, fill):
    """The pages' pad failure: NaN/Inf outside a segment must not reach it -- bit-identical output."""
    wl = W.random_packed(9, [200, 131, 256, 5], heads=2, head_dim=128, capacity=640)
    d = _to(dev, wl)
    base = h3.varlen_attn_fwd(d["q"], d["k"], d["v"], d["cu"], 256)
    cu = wl.cu_seqlens
    for g in range(len(cu) - 1):
        a, b = int(cu[g]), int(cu[g + 1])
        q, k, v = (t.clone() for t in (d["q"], d["k"], d["v"]))
        for t in (q, k, v):
            t[:a] = fill
            t[b:] = fill
        o = h3.varlen_attn_fwd(q, k, v, d["cu"], 256)
        torch.cuda.synchronize()
        assert torch.equal(o[a:b], base[a:b]), f"segment {g} changed under fill {fill}"


def test_rope_in_place_equals_out_of_place(h3, dev):
    wl = W.continuation_batch()
    d = _to(dev, wl)
    qr, kr = _run_rope(h3, d, wl)
    q2, k2 = d["q"].clone(), d["k"].clone()
    h3.rope_apply(q2, k2, d["pos"], d["tag"], d["cu_req"], d["frames"])
    torch.cuda.synchronize()
    assert torch.equal(q2, qr) and torch.equal(k2, kr)


def test_uniform_time_shift_leaves_attention_unchanged(h3, dev):
    """End-to-end invariant: shifting a whole request's time axis does not change its attention."""
    wl = W.tiny_example()
    d = _to(dev, wl)
    outs = []
    for s in (0.0, 238.0):
        frames = torch.tensor([s], device=dev)
        qr, kr = torch.empty_like(d["q"]), torch.empty_like(d["k"])
        h3.rope_apply(d["q"], d["k"], d["pos"], d["tag"], d["cu_req"], frames, q_out=qr, k_out=kr)
        outs.append(h3.varlen_attn_fwd(qr, kr, d["v"], d["cu"], 20).float())
    assert (outs[0] - outs[1]).abs().max().item() <= 2e-2


@pytest.mark.parametrize("cu,maxs,cap", [([0, 30, 20, 45], 30, 64),    # decreasing
                                         ([0, 10, 30, 70], 40, 64),    # beyond capacity
                                         ([5, 10, 30, 45], 25, 64),    # not 0-based
                                         ([0, 10, 300, 345], 128, 400)])  # longer than max_seqlen
def test_bad_cu_seqlens_are_reported_not_followed(h3, dev, cu, maxs, cap):
    wl = W.random_packed(3, [cap], heads=2, head_dim=64)
    d = _to(dev, wl)
    o = torch.full_like(d["q"], 9.0)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=dev)
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], cu_t, maxs, out=o)
    assert h3.get_device_error(dev) == 3  # H3_ERR_BAD_CU_SEQLENS
    assert h3.get_device_error(dev) == 0  # cleared by the read


def test_all_segments_empty(h3, dev):
    wl = W.random_packed(4, [64], heads=2, head_dim=64)
    d = _to(dev, wl)
    o = torch.full_like(d["q"], 2.0)
    cu_t = torch.zeros(4, dtype=torch.int32, device=dev)
    h3.varlen_attn_fwd(d["q"], d["k"], d["v"], cu_t, 1, out=o)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    assert torch.all(o == 2.0)


# ---------------------------------------------------------------------------------------------
# window partition (the shifted 3D window workload: 32x48x84 grid, 4x8x8 windows)
# ---------------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def window_case():
    return W.window_grid()


@pytest.mark.parametrize("layer", [0, 1])
def test_window_pack_is_exact(h3, dev, window_case, layer):
    wl = window_case
    shift = wl.shift if wl.layer_shifted[layer] else (0, 0, 0)
    q, k, v = (t.to(dev) for t in wl.layers[layer])
    perm, cu, (qp, kp, vp) = h3.window_pack(wl.grid, wl.window, shift, [q, k, v])
    torch.cuda.synchronize()
    p_ref, cu_ref = oracle.window_partition(wl.grid, wl.window, shift)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(cu.cpu().numpy(), cu_ref)
    assert len(cu_ref) - 1 == (528 if layer == 0 else 693)
    idx = torch.from_numpy(p_ref.astype(np.int64)).to(dev)
    for src, dst in ((q, qp), (k, kp), (v, vp)):
        assert torch.equal(dst, src.index_select(0, idx))  # a gather is a pure copy
    back = h3.window_unpack(perm, vp)
    torch.cuda.synchronize()
    assert torch.equal(back, v)


@pytest.fixture(scope="module", params=[0, 1], ids=["regular", "shifted"])
def window_layer(request, h3, dev, window_case):
    """Both GPU paths of one layer of the 32x48x84 grid -- pack -> varlen attention -> unpack, and
    attention in place on the grid -- and the oracle over every window of the layer."""
    wl, layer = window_case, request.param
    shift = wl.shift if wl.layer_shifted[layer] else (0, 0, 0)
    q, k, v = (t.to(dev) for t in wl.layers[layer])
    perm, cu, (qp, kp, vp) = h3.window_pack(wl.grid, wl.window, shift, [q, k, v])
    op, lsep = h3.varlen_attn_fwd(qp, kp, vp, cu, 256, return_lse=True)
    o_packed = h3.window_unpack(perm, op)
    o_inpl, lse_inpl = h3.window_attn_fwd(q, k, v, wl.grid, wl.window, shift, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    p_ref, cu_ref = oracle.window_partition(wl.grid, wl.window, shift)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    res = dict(layer=layer, perm=p_ref, cu=cu_ref, o_packed=o_packed.cpu(), lse_packed_order=lsep.cpu(),
               o_inpl=o_inpl.cpu(), lse_inpl=lse_inpl.cpu())
    del q, k, v, qp, kp, vp, op, lsep, o_packed, o_inpl, lse_inpl
    torch.cuda.empty_cache()
    # the oracle on every window, a chunk of windows at a time (fp64 from the bf16 inputs)
    qc, kc, vc = wl.layers[layer]
    N, H, D = qc.shape
    ref_o = np.empty((N, H, D), np.float32)   # in packed (window) order
    ref_lse = np.empty((H, N), np.float64)
    nwin = len(cu_ref) - 1
    for w0 in range(0, nwin, 64):
        w1 = min(nwin, w0 + 64)
        a, b = int(cu_ref[w0]), int(cu_ref[w1])
        rows = torch.from_numpy(p_ref[a:b].astype(np.int64))
        chunk = [x[rows].float().numpy().astype(np.float64) for x in (qc, kc, vc)]
        o, l = oracle.varlen_attention(*chunk, cu_ref[w0:w1 + 1] - a)
        ref_o[a:b] = o
        ref_lse[:, a:b] = l
    res["ref_o"], res["ref_lse"] = ref_o, ref_lse
    return res


def test_window_attention_layer_against_oracle(window_layer):
    """pack -> varlen attention over window segments -> unpack, every window of the layer."""
    r = window_layer
    perm = r["perm"].astype(np.int64)
    assert len(r["cu"]) - 1 == (528 if r["layer"] == 0 else 693)
    _close(r["o_packed"][perm].float().numpy(), r["ref_o"], f"windows, packed path, layer {r['layer']}")
    _lse_close(r["lse_packed_order"].numpy(), r["ref_lse"], f"windows, packed path, layer {r['layer']}")


def test_window_attention_in_place_against_oracle_and_packed_path(window_layer):
    """Attention in place on the grid, every window of the layer against the oracle, and every row
    against the packed GPU path (keys are grouped into tiles differently, so the summation order
    differs: the same tolerance)."""
    r = window_layer
    perm = r["perm"].astype(np.int64)
    o_inpl = r["o_inpl"][perm].float().numpy()  # packed order
    _close(o_inpl, r["ref_o"], f"windows in place, layer {r['layer']}")
    _lse_close(r["lse_inpl"][:, perm].numpy(), r["ref_lse"], f"windows in place, layer {r['layer']}")
    _close(r["o_inpl"].float().numpy(), r["o_packed"].float().numpy(),
           f"in place vs packed, layer {r['layer']}")


def test_unpack_reports_bad_perm(h3, dev):
    n = 64
    perm = torch.arange(n, dtype=torch.int32, device=dev)
    perm[5] = n + 3  # out of range: the row is skipped and reported
    src = torch.randn(n, 16, device=dev).to(torch.bfloat16)
    dst = torch.zeros_like(src)
    h3.window_unpack(perm, src, dst)
    assert h3.get_device_error(dev) == 9  # H3_ERR_BAD_PERM
    ok = torch.ones(n, dtype=torch.bool)
    ok[5] = False
    assert torch.equal(dst[ok.to(dev)], src[ok.to(dev)])


# ---------------------------------------------------------------------------------------------
# window attention in place on the grid (no packed copies)
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("grid,win,shift", [((5, 9, 11), (4, 8, 8), (2, 4, 4)),
                                            ((3, 16, 8), (2, 8, 8), (1, 4, 0)),
                                            ((6, 7, 5), (4, 4, 8), (0, 2, 3)),
                                            ((7, 9, 20), (3, 4, 16), (1, 2, 8)),
                                            # odd window height (no half-height maps), one-tile
                                            # windows of 4 frames, cropped frames and columns
                                            ((5, 3, 70), (4, 1, 32), (2, 0, 16)),
                                            # a window wider than the grid: most of every box
                                            # lies outside it; height-2 edge boxes of height 1
                                            ((9, 6, 10), (2, 2, 64), (1, 1, 0))])
def test_window_attention_in_place_small_grids_full_oracle(h3, dev, D, grid, win, shift):
    n = grid[0] * grid[1] * grid[2]
    rng = np.random.default_rng(n + D)
    q, k, v = (torch.from_numpy(rng.standard_normal((n, 3, D)).astype(np.float32)).to(torch.bfloat16)
               for _ in range(3))
    o, lse = h3.window_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, win, shift, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    perm, cu = oracle.window_partition(grid, win, shift)
    ref_o, ref_lse = oracle.varlen_attention(oracle.window_pack(q, perm), oracle.window_pack(k, perm),
                                             oracle.window_pack(v, perm), cu)
    ref_o = oracle.window_unpack(ref_o, perm)
    ref_lse_orig = np.empty_like(ref_lse)
    ref_lse_orig[:, perm] = ref_lse
    _close(o.float().cpu().numpy(), ref_o, f"in place {grid} {win} {shift} D {D}")
    _lse_close(lse.cpu().numpy(), ref_lse_orig, f"in place {grid} {win} {shift} D {D}")


def _random_window_geometry(seed):
    """A seeded random grid and a supported window (height x width dividing 128, at most 256
    tokens) with a random shift: edge windows cropped on every side, windows wider than the grid."""
    rng = np.random.default_rng(seed)
    while True:
        win = (int(rng.choice([1, 2, 3, 4])), int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 2, 4, 8, 16, 32, 64])))
        if 128 % (win[1] * win[2]) == 0 and win[0] * win[1] * win[2] <= 256 and win[1] * win[2] >= 4:
            break
    grid = (int(rng.integers(1, 10)), int(rng.integers(1, 21)), int(rng.integers(1, 41)))
    shift = tuple(int(rng.integers(0, w)) for w in win)
    return grid, win, shift


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("seed", range(6))
def test_window_random_geometries_against_oracle(h3, dev, D, seed):
    """Seeded random grids, windows and shifts: the partition (perm and cu_seqlens) bit-exact, the
    packed rows exact, and attention in place on every row against the oracle."""
    grid, win, shift = _random_window_geometry(2000 + seed)
    n = grid[0] * grid[1] * grid[2]
    rng = np.random.default_rng(2100 + seed + D)
    q, k, v = (torch.from_numpy(rng.standard_normal((n, 2, D)).astype(np.float32)).to(torch.bfloat16)
               for _ in range(3))
    what = f"grid {grid} win {win} shift {shift} D {D}"
    perm_ref, cu_ref = oracle.window_partition(grid, win, shift)
    perm, cu, packed = h3.window_pack(grid, win, shift, [q.to(dev)])
    torch.cuda.synchronize()
    assert np.array_equal(perm.cpu().numpy(), perm_ref), what
    assert np.array_equal(cu.cpu().numpy(), cu_ref), what
    assert torch.equal(packed[0].cpu(), oracle.window_pack(q, perm_ref)), what
    o, lse = h3.window_attn_fwd(q.to(dev), k.to(dev), v.to(dev), grid, win, shift, return_lse=True)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    ref_o, ref_lse = oracle.varlen_attention(oracle.window_pack(q, perm_ref), oracle.window_pack(k, perm_ref),
                                             oracle.window_pack(v, perm_ref), cu_ref)
    ref_o = oracle.window_unpack(ref_o, perm_ref)
    ref_lse_orig = np.empty_like(ref_lse)
    ref_lse_orig[:, perm_ref] = ref_lse
    _close(o.float().cpu().numpy(), ref_o, what)
    _lse_close(lse.cpu().numpy(), ref_lse_orig, what)


def test_cuda_graph_replay_is_bit_identical_to_eager(h3, dev):
    """RoPE + varlen attention captured once in a CUDA graph and replayed on new inputs (copied
    into the captured buffers) give the same bytes as eager calls."""
    wl = W.tiny_example(capacity=64)
    d = _to(dev, wl)
    H, D = wl.num_heads, wl.head_dim
    ws = torch.empty(max(16, h3.varlen_attn_workspace_size(wl.num_segments, H, wl.max_seqlen, D)),
                     dtype=torch.uint8, device=dev)
    qr, kr, o = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["q"])
    q_in, k_in, v_in = d["q"].clone(), d["k"].clone(), d["v"].clone()

    def step():
        h3.rope_apply(q_in, k_in, d["pos"], d["tag"], d["cu_req"], d["frames"], num_tokens=wl.num_tokens,
                      q_out=qr, k_out=kr)
        h3.varlen_attn_fwd(qr, kr, v_in, d["cu"], wl.max_seqlen, out=o, workspace=ws)

    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        step()                                    # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    gen = torch.Generator().manual_seed(9)
    for _ in range(3):
        for t in (q_in, k_in, v_in):
            t.copy_(torch.randn(t.shape, generator=gen).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        got = o.clone()
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        assert torch.equal(got[:wl.num_tokens], o[:wl.num_tokens])
    assert h3.get_device_error(dev) == 0
