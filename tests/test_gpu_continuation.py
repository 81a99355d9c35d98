"""GPU parity of the continuation-window kernels through the C ABI, against the oracle.

Packing, append and the target-only update move bytes, so they are compared bit for bit
(positions, tags and target mask included).  The chain into RoPE -- the packed rows rotated with
the plan's start frame -- is compared with the fp64 oracle at the RoPE tolerance.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


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


def _rows(rng, n, row_bytes):
    return torch.from_numpy(rng.integers(-2 ** 31, 2 ** 31 - 1, size=(n, row_bytes // 4)).astype(np.int32))


# (text, clip frames, clip audio, frame h, frame w, new frames, new audio, tail, frames/latent, row bytes)
CASES = [
    (5, 29, 200, 2, 3, 29, 200, 7, 4, 64),       # H3-like proportions
    (0, 7, 0, 1, 1, 7, 0, 7, 4, 16),             # no text, no audio, tail = whole clip
    (3, 40, 9, 2, 2, 9, 30, 7, 4, 32),           # audio shorter than the cut: no audio tail
    (5, 245, 500, 2, 3, 20, 150, 7, 1, 48),      # the printed start frame 238
    (11, 12, 77, 3, 5, 30, 91, 3, 2, 80),        # another tail length
]


def _sources(case, seed):
    text, cf, ca, fh, fw, nf, na, tail, fpl, rb = case
    rng = np.random.default_rng(seed)
    hw = fh * fw
    return (_rows(rng, text, rb), _rows(rng, cf * hw, rb), _rows(rng, ca, rb), _rows(rng, nf * hw, rb),
            _rows(rng, na, rb))


@pytest.mark.parametrize("case", CASES)
def test_pack_is_bit_exact(h3, dev, case):
    text, cf, ca, fh, fw, nf, na, tail, fpl, rb = case
    cfg = h3.continuation_config(text, cf, ca, fh, fw, nf, na, tail, fpl)
    src = _sources(case, seed=sum(case))
    rows, pos, tag, target = h3.continuation_pack(cfg, *[t.to(dev) if t.shape[0] else None for t in src])
    torch.cuda.synchronize()
    plan = oracle.continuation_plan(text, cf, ca, fh, fw, nf, na, tail_frames=tail, frames_per_latent=fpl)
    r, p, tg, tgt = oracle.continuation_pack(plan, *[t.numpy() for t in src], fh, fw)
    assert np.array_equal(rows.cpu().numpy(), r)
    assert np.array_equal(pos.cpu().numpy(), p)
    assert np.array_equal(tag.cpu().numpy(), tg) and np.array_equal(target.cpu().numpy(), tgt)


@pytest.mark.parametrize("case", CASES)
def test_append_is_bit_exact_and_leaves_the_clip_untouched(h3, dev, case):
    text, cf, ca, fh, fw, nf, na, tail, fpl, rb = case
    hw = fh * fw
    cfg = h3.continuation_config(text, cf, ca, fh, fw, nf, na, tail, fpl)
    _, clip_v, clip_a, new_v, new_a = _sources(case, seed=3 * sum(case))
    plan = oracle.continuation_plan(text, cf, ca, fh, fw, nf, na, tail_frames=tail, frames_per_latent=fpl)
    # clip buffers with room for the result plus 3 sentinel rows that must stay untouched
    sent = torch.full((3, rb // 4), 0x5A5A5A5A, dtype=torch.int32)
    buf_v = torch.cat([clip_v, torch.zeros((plan.out_video_frames * hw - cf * hw, rb // 4), dtype=torch.int32), sent])
    buf_a = torch.cat([clip_a, torch.zeros((plan.out_audio_rows - ca, rb // 4), dtype=torch.int32), sent])
    dv, da = buf_v.to(dev), buf_a.to(dev)
    h3.continuation_append(cfg, new_v.to(dev), new_a.to(dev), dv, da)
    torch.cuda.synchronize()
    v, a = oracle.continuation_append(plan, clip_v.numpy(), clip_a.numpy(), new_v.numpy(), new_a.numpy(), fh, fw)
    got_v, got_a = dv.cpu().numpy(), da.cpu().numpy()
    assert np.array_equal(got_v[:len(v)], v) and np.array_equal(got_a[:len(a)], a)
    assert np.array_equal(got_v[len(v):], sent.numpy()) and np.array_equal(got_a[len(a):], sent.numpy())


def test_masked_row_update_is_bit_exact(h3, dev):
    rng = np.random.default_rng(5)
    x, x_new = _rows(rng, 1000, 96), _rows(rng, 1000, 96)
    mask = torch.from_numpy((rng.random(1000) < 0.4).astype(np.uint8))
    d = x.to(dev)
    h3.masked_row_update(d, x_new.to(dev), mask.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), oracle.masked_update(x.numpy(), x_new.numpy(), mask.numpy()))


def test_h3_shaped_window_packs_bit_exact_and_rotates_with_the_start_frame(h3, dev):
    """The previous window is the H3 request's video (29 latent frames of 40x50) and audio
    (200 rows); the next window has the same shape; rows are 40 heads x 128 bf16."""
    H, D = 40, 128
    case = (558, 29, 200, 40, 50, 29, 200, 7, 4, H * D * 2)
    text, cf, ca, fh, fw, nf, na, tail, fpl, rb = case
    cfg = h3.continuation_config(text, cf, ca, fh, fw, nf, na, tail, fpl)
    rng = np.random.default_rng(41)
    src = [torch.from_numpy(rng.standard_normal((n, H, D)).astype(np.float32)).to(torch.bfloat16)
           for n in (text, cf * fh * fw, ca, nf * fh * fw, na)]
    rows, pos, tag, target = h3.continuation_pack(cfg, *[t.to(dev) for t in src])
    plan = h3.continuation_plan(cfg)
    assert plan.num_rows == 72812 and plan.start_frame == 88 and plan.audio_cut == 146
    ref_plan = oracle.continuation_plan(*case[:7], tail_frames=tail, frames_per_latent=fpl)
    r, p, tg, tgt = oracle.continuation_pack(ref_plan, *[t.view(torch.int16).numpy() for t in src], fh, fw)
    torch.cuda.synchronize()
    assert np.array_equal(rows.view(torch.int16).cpu().numpy(), r)
    assert np.array_equal(pos.cpu().numpy(), p) and np.array_equal(tag.cpu().numpy(), tg)
    assert np.array_equal(target.cpu().numpy(), tgt)
    # RoPE with the continuation shift s * 40 / 24 on the packed rows, one request
    n = plan.num_rows
    cu_req = torch.tensor([0, n], dtype=torch.int32, device=dev)
    frames = torch.tensor([float(plan.start_frame)], dtype=torch.float32, device=dev)
    q_out = torch.empty_like(rows)
    h3.rope_apply(rows, None, pos, tag, cu_req, frames, q_out=q_out)
    torch.cuda.synchronize()
    assert h3.get_device_error(dev) == 0
    sample = np.unique(np.concatenate([np.arange(0, n, 97), plan.group_offset[1:5], [n - 1]]))
    ref = oracle.rope_apply(rows.cpu(), p, tg, np.array([0, n]), np.array([float(plan.start_frame)]),
                            rows=sample)
    err = np.abs(q_out.cpu().float().numpy()[sample] - ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
