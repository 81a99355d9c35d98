"""Continuation window packing -- test infrastructure only, never product code.

Source: [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section
"Crossing the time boundary" (continuation): step 1 takes two reference signals straight from the
previous window's latents -- the last 7 latent time cells of the video, and the audio tail cut at
the global 40 Hz boundary; step 2 concatenates five row groups into one DiT sequence in the order
(1) text / original reference, (2) tail audio reference, (3) tail video reference, (4) new-window
audio noise, (5) new-window video noise; only groups 4 and 5 (targets) are updated by the
denoising steps, groups 2 and 3 stay frozen; step 3 shifts every token's time coordinate by
s * 40 / 24 before RoPE (s = the window's first frame, 24 FPS video, 40 Hz audio).  Afterwards the
part of the new samples that overlaps the reference rows in time is discarded and only the
non-overlapping suffix is appended to the clip.

Readings where the pages leave a step open:
  * Units.  Video latents have `frames_per_latent` video frames (24 FPS) per latent frame
    (4 makes the H3 request's 29 latent frames and 200 audio rows one 5 s window); audio latents
    are 40 Hz rows.  The new window starts where the video tail starts: g0 = clip_frames - 7
    latent frames, s = g0 * frames_per_latent video frames.
  * The 40 Hz boundary: the audio tail starts at the 40 Hz row containing time s / 24 s,
    audio_cut = floor(s * 40 / 24) (the printed example s = 238 -> 396.67 -> row 396).
  * Positions are local to the new window (its first frame and audio row at t = 0); the shift
    s * 40 / 24 is added by RoPE to every row.  Text rows t = 0.. (own position space); the audio
    tail t = 0.. from audio_cut; the video tail t = 0..6 with (h, w) of the latent grid; the new
    audio t = 0..; the new video t = 0.. with (h, w).  So reference and target rows that share a
    moment share a time coordinate.
  * Overlap: the new window's first 7 latent frames coincide with the video tail, its first
    (clip_audio_rows - audio_cut) audio rows with the audio tail; those are discarded, the rest
    appended: the clip grows to g0 + new_frames latent frames and audio_cut + new_audio_rows rows.
  * Attention segments: the request is one segment over all five groups (the targets must read
    the tails, and in the printed order a modality's tail and targets are not adjacent).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TAG_TEXT, TAG_VIDEO, TAG_AUDIO = 0, 1, 2


@dataclass
class ContinuationPlan:
    tail_start: int          # g0: first latent frame of the video tail (global)
    start_frame: int         # s = g0 * frames_per_latent, in 24 FPS video frames
    audio_cut: int           # first audio row of the tail (global 40 Hz index)
    group_rows: tuple        # rows of the 5 groups in packed order
    group_offset: tuple      # exclusive prefix, length 6
    num_rows: int
    keep_video_from: int     # first new latent frame appended to the clip
    keep_audio_from: int     # first new audio row appended
    out_video_frames: int
    out_audio_rows: int


def continuation_plan(text_rows, clip_video_frames, clip_audio_rows, frame_h, frame_w,
                      new_video_frames, new_audio_rows, tail_frames=7, frames_per_latent=4):
    g0 = clip_video_frames - tail_frames
    if g0 < 0 or new_video_frames < tail_frames:
        raise ValueError("the clip and the new window need at least tail_frames latent frames")
    s = g0 * frames_per_latent
    audio_cut = min((s * 40) // 24, clip_audio_rows)     # floor(s * 40 / 24), inside the clip
    ref_audio = clip_audio_rows - audio_cut
    if new_audio_rows < ref_audio:
        raise ValueError("the new window's audio must cover the audio tail")
    hw = frame_h * frame_w
    rows = (text_rows, ref_audio, tail_frames * hw, new_audio_rows, new_video_frames * hw)
    off = tuple(int(x) for x in np.concatenate([[0], np.cumsum(rows)]))
    return ContinuationPlan(tail_start=g0, start_frame=s, audio_cut=audio_cut, group_rows=rows,
                            group_offset=off, num_rows=off[5], keep_video_from=tail_frames,
                            keep_audio_from=ref_audio, out_video_frames=g0 + new_video_frames,
                            out_audio_rows=audio_cut + new_audio_rows)


def continuation_pack(plan, text, clip_video, clip_audio, new_video, new_audio, frame_h, frame_w):
    """Rows [num_rows, ...] in the five-group order, positions fp32 [num_rows, 3], tags u8 and
    the target mask u8 (1 on groups 4 and 5).  clip_video / new_video are [frames*H*W, ...] in
    row-major (t, h, w) order; clip_audio / new_audio [rows, ...]."""
    hw = frame_h * frame_w
    tail_frames = plan.keep_video_from
    tail_v = np.asarray(clip_video)[plan.tail_start * hw:(plan.tail_start + tail_frames) * hw]
    tail_a = np.asarray(clip_audio)[plan.audio_cut:plan.audio_cut + plan.group_rows[1]]
    rows = np.concatenate([np.asarray(text), tail_a, tail_v, np.asarray(new_audio),
                           np.asarray(new_video)])

    def seq(n):
        p = np.zeros((n, 3), np.float32)
        p[:, 0] = np.arange(n)
        return p

    def grid(frames):
        t, h, w = np.meshgrid(np.arange(frames), np.arange(frame_h), np.arange(frame_w), indexing="ij")
        return np.stack([t.reshape(-1), h.reshape(-1), w.reshape(-1)], 1).astype(np.float32)

    pos = np.concatenate([seq(plan.group_rows[0]), seq(plan.group_rows[1]), grid(tail_frames),
                          seq(plan.group_rows[3]), grid(plan.group_rows[4] // hw)])
    tag = np.concatenate([np.full(plan.group_rows[0], TAG_TEXT), np.full(plan.group_rows[1], TAG_AUDIO),
                          np.full(plan.group_rows[2], TAG_VIDEO), np.full(plan.group_rows[3], TAG_AUDIO),
                          np.full(plan.group_rows[4], TAG_VIDEO)]).astype(np.uint8)
    target = np.concatenate([np.zeros(plan.group_offset[3], np.uint8),
                             np.ones(plan.num_rows - plan.group_offset[3], np.uint8)])
    return rows, pos, tag, target


def continuation_append(plan, clip_video, clip_audio, new_video, new_audio, frame_h, frame_w):
    """The clip after the window: every existing row (the overlap keeps the earlier result), then
    the new rows past the overlap."""
    hw = frame_h * frame_w
    video = np.concatenate([np.asarray(clip_video), np.asarray(new_video)[plan.keep_video_from * hw:]])
    audio = np.concatenate([np.asarray(clip_audio), np.asarray(new_audio)[plan.keep_audio_from:]])
    return video, audio


def masked_update(x, x_new, target):
    """One denoising update that touches only the target rows."""
    out = np.array(x, copy=True)
    m = np.asarray(target).astype(bool)
    out[m] = np.asarray(x_new)[m]
    return out
