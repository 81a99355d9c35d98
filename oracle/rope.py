"""fp64 modality-tagged rotary position encoding with the continuation time shift.

Test infrastructure only, never product code.

Sources:
  [H3-vLLM] §3 "Packed sequence and modality identity", causal chain item 1: each token
      carries a discrete modality tag (text / video / audio) that selects its RoPE
      frequencies; the position spaces of the modalities are independent.  The stage table
      records spatial/temporal positions per row.
  [H3-fast] "Crossing the time boundary", step 3: before RoPE, the time coordinate is moved
      to t_global = t_local + s * 40/24 (s = the window's start frame; 40 Hz audio, 24 fps
      video); only the time axis moves, spatial coordinates stay; decimals are kept
      (start frame 238 -> 396.67).

Readings where the pages are silent:
  * Rotation: pairs (x[2i], x[2i+1]) rotated by angle phi_i, as in the original RoFormer
    formulation:  x'[2i] = x[2i] cos phi - x[2i+1] sin phi,  x'[2i+1] = x[2i] sin phi + x[2i+1] cos phi.
  * Frequency ladder of a band of width d: theta_i = base^(-2i/d), i in [0, d/2).
  * Text and audio: one band over all D dims driven by t.  Video: three bands,
    dims [0, d_t) by t, [d_t, d_t + d_h) by h, [d_t + d_h, D) by w, each with its own ladder;
    default split D/2 : D/4 : D/4 (32/16/16 at D = 64), base 10000 for every modality.
  * The time shift applies to every token of the request (its time coordinate only).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import numpy as np

TAG_TEXT, TAG_VIDEO, TAG_AUDIO = 0, 1, 2


def continuation_time_shift(start_frame: float, audio_hz: float = 40.0, video_fps: float = 24.0) -> float:
    """s * 40/24: the amount added to the time coordinate of a continuation window ([H3-fast])."""
    return float(start_frame) * float(audio_hz) / float(video_fps)


def video_axis_split(head_dim: int, dims_t: int = 0, dims_h: int = 0, dims_w: int = 0) -> Tuple[int, int, int]:
    """(d_t, d_h, d_w); zeros select the default D/2 : D/4 : D/4."""
    if dims_t == 0 and dims_h == 0 and dims_w == 0:
        return head_dim // 2, head_dim // 4, head_dim // 4
    assert dims_t + dims_h + dims_w == head_dim
    return dims_t, dims_h, dims_w


def rope_inv_freq(base: float, band_dims: int) -> np.ndarray:
    """theta_i = base^(-2i/d) for i in [0, d/2), fp64."""
    i = np.arange(band_dims // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / float(band_dims))


@dataclass
class RopeConfig:
    base_text: float = 10000.0
    base_video: float = 10000.0
    base_audio: float = 10000.0
    video_dims_t: int = 0
    video_dims_h: int = 0
    video_dims_w: int = 0
    audio_hz: float = 40.0
    video_fps: float = 24.0


def rope_angles(pos: np.ndarray, tag: np.ndarray, head_dim: int, cfg: Optional[RopeConfig] = None,
                time_offset: Optional[np.ndarray] = None) -> np.ndarray:
    """Angles phi [N, D/2] in fp64 for each token's D/2 rotation pairs.

    pos: [N, 3] local (t, h, w); tag: [N]; time_offset: [N] added to t (already s*40/24).
    """
    cfg = cfg or RopeConfig()
    pos = np.asarray(pos, dtype=np.float64)
    tag = np.asarray(tag)
    N = pos.shape[0]
    t = pos[:, 0].copy()
    if time_offset is not None:
        t = t + np.asarray(time_offset, dtype=np.float64)
    h, w = pos[:, 1], pos[:, 2]
    P = head_dim // 2
    phi = np.zeros((N, P), dtype=np.float64)
    dt, dh, dw = video_axis_split(head_dim, cfg.video_dims_t, cfg.video_dims_h, cfg.video_dims_w)
    vid = tag == TAG_VIDEO
    aud = tag == TAG_AUDIO
    txt = ~(vid | aud)
    # video: three bands, each with its own ladder, driven by t, h and w
    phi[vid, 0:dt // 2] = np.outer(t[vid], rope_inv_freq(cfg.base_video, dt))
    phi[vid, dt // 2:(dt + dh) // 2] = np.outer(h[vid], rope_inv_freq(cfg.base_video, dh))
    phi[vid, (dt + dh) // 2:P] = np.outer(w[vid], rope_inv_freq(cfg.base_video, dw))
    # text and audio: one band over all D dims, driven by t
    phi[txt, :] = np.outer(t[txt], rope_inv_freq(cfg.base_text, head_dim))
    phi[aud, :] = np.outer(t[aud], rope_inv_freq(cfg.base_audio, head_dim))
    return phi


def rotate_pairs(x: np.ndarray, phi: np.ndarray) -> np.ndarray:
    """Rotate (x[..., 2i], x[..., 2i+1]) by phi[..., i].  x: [N, H, D]; phi: [N, D/2]."""
    x = np.asarray(x, dtype=np.float64)
    c = np.cos(phi)[:, None, :]
    s = np.sin(phi)[:, None, :]
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def request_time_offsets(n_tokens: int, cu_requests: Optional[Sequence[int]],
                         start_frames: Optional[Sequence[float]], cfg: Optional[RopeConfig] = None) -> np.ndarray:
    """Per-token s_r * 40/24 for the request r that owns the token (zero without requests)."""
    cfg = cfg or RopeConfig()
    off = np.zeros(n_tokens, dtype=np.float64)
    if cu_requests is None or start_frames is None:
        return off
    cu = np.asarray(cu_requests, dtype=np.int64)
    for r in range(len(cu) - 1):
        off[cu[r]:cu[r + 1]] = continuation_time_shift(start_frames[r], cfg.audio_hz, cfg.video_fps)
    return off


def rope_apply(x, pos, tag, cu_requests=None, start_frames=None, cfg: Optional[RopeConfig] = None,
               num_tokens: Optional[int] = None, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Tagged RoPE of x [C, H, D] for the first num_tokens rows (rest returned as NaN).

    cu_requests [R+1] / start_frames [R]: continuation requests packed in the sequence; each
    token's time coordinate is shifted by its request's s * 40/24 before the rotation.
    rows: optional subset of row indices (< num_tokens) to evaluate; the result then has
    len(rows) rows, in that order.
    """
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
    if hasattr(x, "detach"):
        x = (x[rows] if rows is not None else x).detach().float().numpy()
    elif rows is not None:
        x = np.asarray(x)[rows]
    x = np.asarray(x, dtype=np.float64)
    C, H, D = x.shape
    if rows is not None:
        n_all = int(np.max(rows)) + 1 if rows.size else 0
        off = request_time_offsets(n_all, cu_requests, start_frames, cfg)[rows]
        phi = rope_angles(np.asarray(pos)[rows], np.asarray(tag)[rows], D, cfg, off)
        return rotate_pairs(x, phi)
    n = C if num_tokens is None else int(num_tokens)
    off = request_time_offsets(n, cu_requests, start_frames, cfg)
    phi = rope_angles(np.asarray(pos)[:n], np.asarray(tag)[:n], D, cfg, off)
    out = np.full_like(x, np.nan)
    out[:n] = rotate_pairs(x[:n], phi)
    return out
