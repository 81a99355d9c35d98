"""Pins for the continuation-window packing oracle, no GPU.

Rows carry labels of their global time (video: global latent frame, audio: global 40 Hz row),
so the tests can check the pages' statements directly: the tail is the last 7 latent frames, the
audio tail starts on the 40 Hz boundary of the tail's start, the five groups come in the printed
order, only targets are updated, and after the overlap is discarded the clip's timeline runs on
without a gap or a repeat.  Source: [H3-fast] "Breaking the engineering bottlenecks of
video-generation models", section "Crossing the time boundary".
"""
import json
import math
import os

import numpy as np
import pytest

import oracle


def _clip(frames, audio, hw, c=4, offset=0):
    """Video rows labelled (global frame, h*w index, 0, 0...), audio rows (global row, -1, ...)."""
    v = np.zeros((frames * hw, c))
    v[:, 0] = np.repeat(np.arange(frames) + offset, hw)
    v[:, 1] = np.tile(np.arange(hw), frames)
    a = np.zeros((audio, c))
    a[:, 0] = np.arange(audio)
    a[:, 1] = -1
    return v, a


def test_printed_start_frame_gives_the_40hz_cut(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "continuation_time_shift.json")))
    s = g["start_frame"]
    shift = s * g["audio_hz"] / g["video_fps"]
    assert round(shift, g["printed_decimals"]) == g["printed_offset"]
    # a clip whose 7-frame tail starts at latent frame 238, one video frame per latent frame
    p = oracle.continuation_plan(5, s + 7, 500, 2, 3, 20, 150, tail_frames=7, frames_per_latent=1)
    assert p.tail_start == s and p.start_frame == s
    assert p.audio_cut == math.floor(shift) == 396      # the 40 Hz row holding t = 238 / 24 s
    assert p.keep_audio_from == 500 - 396


def test_h3_shaped_window_closed_forms():
    # previous window = the H3 request's 29 latent frames x 40 x 50 and 200 audio rows (5 s)
    p = oracle.continuation_plan(558, 29, 200, 40, 50, 29, 200)
    assert p.tail_start == 22 and p.start_frame == 88
    assert p.audio_cut == (88 * 40) // 24 == 146
    assert p.group_rows == (558, 54, 7 * 2000, 200, 29 * 2000)
    assert p.num_rows == 558 + 54 + 14000 + 200 + 58000 == 72812
    assert p.out_video_frames == 29 + 29 - 7 and p.out_audio_rows == 146 + 200


@pytest.mark.parametrize("fpl", [1, 4])
@pytest.mark.parametrize("clip_frames,clip_audio,new_frames,new_audio",
                         [(29, 200, 29, 200), (10, 70, 12, 80), (7, 30, 7, 30), (40, 9, 9, 30)])
def test_pack_groups_positions_tags_and_targets(fpl, clip_frames, clip_audio, new_frames, new_audio):
    fh, fw = 2, 3
    hw = fh * fw
    p = oracle.continuation_plan(5, clip_frames, clip_audio, fh, fw, new_frames, new_audio,
                                 frames_per_latent=fpl)
    cv, ca = _clip(clip_frames, clip_audio, hw)
    nv, na = _clip(new_frames, new_audio, hw)
    nv[:, 2], na[:, 2] = 1, 1                          # mark the new window's rows
    text = np.zeros((5, 4))
    text[:, 0] = np.arange(5)
    text[:, 1] = -2
    rows, pos, tag, target = oracle.continuation_pack(p, text, cv, ca, nv, na, fh, fw)
    off = p.group_offset
    assert rows.shape == (p.num_rows, 4) and pos.shape == (p.num_rows, 3)
    # (1) text
    assert np.array_equal(rows[:off[1], 1], np.full(5, -2)) and np.all(tag[:off[1]] == 0)
    # (2) audio tail: the clip's rows from floor(s * 40 / 24) on, local t from 0
    cut = min((p.start_frame * 40) // 24, clip_audio)
    assert np.array_equal(rows[off[1]:off[2], 0], np.arange(cut, clip_audio))
    assert np.all(rows[off[1]:off[2], 2] == 0) and np.all(tag[off[1]:off[2]] == 2)
    assert np.array_equal(pos[off[1]:off[2], 0], np.arange(clip_audio - cut))
    # (3) video tail: the clip's last 7 latent frames, local t 0..6 with the frame's (h, w)
    assert np.array_equal(rows[off[2]:off[3], 0], np.repeat(np.arange(clip_frames - 7, clip_frames), hw))
    assert np.array_equal(pos[off[2]:off[3], 0], np.repeat(np.arange(7), hw))
    assert np.array_equal(pos[off[2]:off[3], 1] * fw + pos[off[2]:off[3], 2], np.tile(np.arange(hw), 7))
    assert np.all(tag[off[2]:off[3]] == 1)
    # (4) new audio, (5) new video: the new window, local positions from 0, the only targets
    assert np.all(rows[off[3]:, 2] == 1) and np.all(rows[:off[3], 2] == 0)
    assert np.array_equal(pos[off[3]:off[4], 0], np.arange(new_audio)) and np.all(tag[off[3]:off[4]] == 2)
    assert np.array_equal(pos[off[4]:, 0], np.repeat(np.arange(new_frames), hw)) and np.all(tag[off[4]:] == 1)
    assert np.array_equal(target, (np.arange(p.num_rows) >= off[3]).astype(np.uint8))
    # reference and target rows that share a moment share a time coordinate: the tail's frame
    # g0 + t is the new window's frame t
    assert np.array_equal(pos[off[2]:off[3]], pos[off[4]:off[4] + 7 * hw])


@pytest.mark.parametrize("fpl", [1, 4])
@pytest.mark.parametrize("clip_frames,clip_audio,new_frames,new_audio",
                         [(29, 200, 29, 200), (10, 70, 12, 80), (7, 30, 7, 30)])
def test_append_continues_the_timeline_without_gap_or_repeat(fpl, clip_frames, clip_audio, new_frames,
                                                             new_audio):
    fh, fw = 2, 3
    hw = fh * fw
    p = oracle.continuation_plan(5, clip_frames, clip_audio, fh, fw, new_frames, new_audio,
                                 frames_per_latent=fpl)
    cv, ca = _clip(clip_frames, clip_audio, hw)
    # the new window's rows carry their global time: video from the tail start, audio from the cut
    nv, na = _clip(new_frames, new_audio, hw, offset=0)
    nv[:, 0] += p.tail_start
    na[:, 0] += p.audio_cut
    nv[:, 2], na[:, 2] = 1, 1
    v, a = oracle.continuation_append(p, cv, ca, nv, na, fh, fw)
    assert len(v) == p.out_video_frames * hw and len(a) == p.out_audio_rows
    assert np.array_equal(v[:, 0], np.repeat(np.arange(p.out_video_frames), hw))
    assert np.array_equal(a[:, 0], np.arange(p.out_audio_rows))
    # the overlap keeps the earlier result: no new row lands before the clip's end
    assert np.all(v[:clip_frames * hw, 2] == 0) and np.all(v[clip_frames * hw:, 2] == 1)
    assert np.all(a[:clip_audio, 2] == 0) and np.all(a[clip_audio:, 2] == 1)


def test_plan_rejects_windows_shorter_than_the_tail():
    with pytest.raises(ValueError):
        oracle.continuation_plan(5, 6, 40, 2, 2, 10, 40)
    with pytest.raises(ValueError):
        oracle.continuation_plan(5, 10, 40, 2, 2, 6, 40)
    with pytest.raises(ValueError):   # new audio shorter than the audio tail it overlaps
        oracle.continuation_plan(5, 29, 200, 2, 2, 29, 10)


def test_masked_update_touches_only_targets():
    rng = np.random.default_rng(3)
    x, x_new = rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    target = (np.arange(50) >= 20).astype(np.uint8)
    y = oracle.masked_update(x, x_new, target)
    assert np.array_equal(y[:20], x[:20]) and np.array_equal(y[20:], x_new[20:])
