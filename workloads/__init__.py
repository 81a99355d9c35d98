"""Seeded synthetic inputs shaped like the MiniMax-H3 / SeedVR2 attention workloads.

This module only *draws* inputs: Q/K/V values, per-token positions, modality tags, the
packing layout (segment lengths -> cu_seqlens) and per-request continuation start frames.
It holds none of the method's arithmetic (no rotation, no time-shift formula, no softmax,
no window partition).  Both the CPU oracle and the CUDA path are fed from here, and
nothing here imports either of them.

Shapes follow the pages:
  * packed request of 58,758 tokens = text 558 + audio 200 + video 29x40x50
    ("MiniMax-H3 x vLLM-Omni", section 1 "unified architecture", stage table; section 6
    "trim padding", 58,816 aligned vs 58,758 valid);
  * the cu_seqlens worked example [0,10,30,45] (same page, section 3, "minimal example");
  * continuation requests whose time axis is shifted by the start frame s
    ("MiniMax H3 fast and strong", continuation, step 3 "RoPE global time alignment");
  * a 3D latent grid cut into (shifted) windows (same page, "window-aligned SP");
  * the same grid attended block-sparsely over 4x4x4 blocks (same page, "VSA"); the pages give
    no top-k ratio, the default keeps 1/8 of the blocks.

Modality tags: 0 = text, 1 = video, 2 = audio.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np
import torch

TAG_TEXT = 0
TAG_VIDEO = 1
TAG_AUDIO = 2


@dataclass
class PackedWorkload:
    """One packed sequence (possibly several requests) ready for RoPE + varlen attention."""

    name: str
    num_heads: int
    head_dim: int
    q: torch.Tensor  # bf16 [C, H, D] (rows >= N are padding)
    k: torch.Tensor
    v: torch.Tensor
    pos: np.ndarray  # float32 [C, 3]: local (t, h, w); h = w = 0 for text/audio
    tag: np.ndarray  # uint8 [C]
    cu_seqlens: np.ndarray  # int32 [S+1]
    cu_requests: np.ndarray  # int32 [R+1]
    start_frames: np.ndarray  # float32 [R]: continuation window start frame s per request
    capacity: int  # C >= N = cu_seqlens[-1]
    seg_kinds: List[str] = field(default_factory=list)

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_segments(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def max_seqlen(self) -> int:
        return int(np.max(np.diff(self.cu_seqlens))) if self.num_segments else 0

    def attention_flops(self) -> float:
        """4 * H * D * sum(n_g^2): QK^T and PV, in-segment work only."""
        n = np.diff(self.cu_seqlens).astype(np.float64)
        return float(4.0 * self.num_heads * self.head_dim * np.sum(n * n))


@dataclass
class WindowWorkload:
    """A 3D latent grid (T, H, W) in row-major token order, attended in (shifted) windows."""

    name: str
    num_heads: int
    head_dim: int
    grid: Tuple[int, int, int]
    window: Tuple[int, int, int]
    shift: Tuple[int, int, int]
    layers: List[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]]  # per layer (q, k, v) bf16 [N, H, D]
    layer_shifted: List[bool]

    @property
    def num_tokens(self) -> int:
        t, h, w = self.grid
        return t * h * w


def _normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return torch.from_numpy(x).to(torch.bfloat16)


def _text_positions(n: int) -> np.ndarray:
    p = np.zeros((n, 3), dtype=np.float32)
    p[:, 0] = np.arange(n, dtype=np.float32)
    return p


def _video_positions(n: int, frame_h: int, frame_w: int) -> np.ndarray:
    """Row-major (t, h, w) over a frame_h x frame_w patch grid; the last frame may be partial."""
    idx = np.arange(n, dtype=np.int64)
    per = frame_h * frame_w
    p = np.zeros((n, 3), dtype=np.float32)
    p[:, 0] = idx // per
    p[:, 1] = (idx % per) // frame_w
    p[:, 2] = idx % frame_w
    return p


def _assemble(name, seed, H, D, parts, cu_requests, start_frames, capacity=None, scale=1.0,
              pad_fill=float("nan")) -> PackedWorkload:
    """parts: list of (kind, n, positions[n,3], tag) in packing order; one segment each."""
    lens = [n for _, n, _, _ in parts]
    N = int(sum(lens))
    C = N if capacity is None else int(capacity)
    assert C >= N
    cu = np.zeros(len(parts) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    pos = np.zeros((C, 3), dtype=np.float32)
    tag = np.zeros((C,), dtype=np.uint8)
    off = 0
    for _, n, p, tg in parts:
        pos[off:off + n] = p
        tag[off:off + n] = tg
        off += n
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (C, H, D), scale)
    k = _normal_bf16(rng, (C, H, D), scale)
    v = _normal_bf16(rng, (C, H, D), scale)
    if C > N:
        for t in (q, k, v):
            t[N:] = pad_fill
    return PackedWorkload(name=name, num_heads=H, head_dim=D, q=q, k=k, v=v, pos=pos, tag=tag,
                          cu_seqlens=cu, cu_requests=np.asarray(cu_requests, dtype=np.int32),
                          start_frames=np.asarray(start_frames, dtype=np.float32), capacity=C,
                          seg_kinds=[kind for kind, _, _, _ in parts])


def tiny_example(seed: int = 1, capacity: Optional[int] = None) -> PackedWorkload:
    """The pages' worked example: 10 text + 20 video (1x4x5) + 15 audio, cu_seqlens [0,10,30,45].

    2 heads x head_dim 64, Q/K/V ~ N(0,1) rounded to bf16.
    """
    parts = [("text", 10, _text_positions(10), TAG_TEXT),
             ("video", 20, _video_positions(20, 4, 5), TAG_VIDEO),
             ("audio", 15, _text_positions(15), TAG_AUDIO)]
    return _assemble("tiny_example_45tok_2x64", seed, 2, 64, parts, [0, 45], [0.0], capacity)


def single_request_4k(seed: int = 2, capacity: Optional[int] = None) -> PackedWorkload:
    """4,096 tokens: text 256 + audio 320 (40 Hz x 8 s) + video 11x16x20; 24 x 128.

    Q/K/V drawn N(0,1) and multiplied by 1/sqrt(128) before rounding to bf16.
    """
    parts = [("text", 256, _text_positions(256), TAG_TEXT),
             ("audio", 320, _text_positions(320), TAG_AUDIO),
             ("video", 3520, _video_positions(3520, 16, 20), TAG_VIDEO)]
    return _assemble("single_request_4096tok_24x128", seed, 24, 128, parts, [0, 4096], [0.0],
                     capacity, scale=1.0 / np.sqrt(128.0))


def h3_full_request(seed: int = 3, capacity: Optional[int] = 58816) -> PackedWorkload:
    """58,758 tokens: text 558 + audio 200 (40 Hz x 5 s) + video 29x40x50; 40 x 128.

    Default capacity 58,816 (the aligned length the pages quote) with NaN-filled pad rows.
    """
    parts = [("text", 558, _text_positions(558), TAG_TEXT),
             ("audio", 200, _text_positions(200), TAG_AUDIO),
             ("video", 58000, _video_positions(58000, 40, 50), TAG_VIDEO)]
    return _assemble("h3_request_58758tok_40x128", seed, 40, 128, parts, [0, 58758], [0.0], capacity)


CONTINUATION_START_FRAMES = (0.0, 119.0, 238.0, 357.0)


def continuation_lengths(seed: int = 4) -> List[Tuple[int, int, int]]:
    """Per-request (text, audio, video) lengths: L ~ U{8000..20000}; text 2 %, audio 3 %, video rest."""
    rng = np.random.default_rng(seed)
    L = rng.integers(8000, 20001, size=4)
    out = []
    for l in L:
        l = int(l)
        text = (2 * l) // 100
        audio = (3 * l) // 100
        out.append((text, audio, l - text - audio))
    return out


def continuation_batch(seed: int = 4, capacity: Optional[int] = None,
                       per_request_segments: bool = False) -> PackedWorkload:
    """4 continuation requests packed back to back, each [text | audio | video].

    By default each modality of each request is its own segment (12 segments).  With
    ``per_request_segments`` each request is one segment (4 segments).  Video rows fill a
    40x50 patch grid per latent frame, row-major.  Request r starts at frame s_r.
    """
    lens = continuation_lengths(seed)
    parts = []
    cu_req = [0]
    for (text, audio, video) in lens:
        parts.append(("text", text, _text_positions(text), TAG_TEXT))
        parts.append(("audio", audio, _text_positions(audio), TAG_AUDIO))
        parts.append(("video", video, _video_positions(video, 40, 50), TAG_VIDEO))
        cu_req.append(cu_req[-1] + text + audio + video)
    wl = _assemble("continuation_4req_40x128", seed, 40, 128, parts, cu_req,
                   list(CONTINUATION_START_FRAMES), capacity)
    if per_request_segments:
        wl.cu_seqlens = np.asarray(cu_req, dtype=np.int32)
        wl.seg_kinds = ["request"] * 4
        wl.name = "continuation_4req_4seg_40x128"
    return wl


def window_grid(seed: int = 5, grid=(32, 48, 84), window=(4, 8, 8), shift=(2, 4, 4),
                heads: int = 24, head_dim: int = 128, num_layers: int = 2) -> WindowWorkload:
    """Latent grid in row-major (t, h, w) order; layers alternate unshifted / shifted windows.

    Each layer gets its own Q/K/V ~ N(0,1) in bf16.
    """
    rng = np.random.default_rng(seed)
    n = grid[0] * grid[1] * grid[2]
    layers = []
    for _ in range(num_layers):
        layers.append((_normal_bf16(rng, (n, heads, head_dim)),
                       _normal_bf16(rng, (n, heads, head_dim)),
                       _normal_bf16(rng, (n, heads, head_dim))))
    return WindowWorkload(name=f"window_{grid[0]}x{grid[1]}x{grid[2]}_w{window[0]}x{window[1]}x{window[2]}",
                          num_heads=heads, head_dim=head_dim, grid=tuple(grid), window=tuple(window),
                          shift=tuple(shift), layers=layers,
                          layer_shifted=[(i % 2) == 1 for i in range(num_layers)])


def random_packed(seed: int, lengths, heads: int, head_dim: int, capacity: Optional[int] = None,
                  scale: float = 1.0, tags=None) -> PackedWorkload:
    """Arbitrary segment lengths (edge cases: empty, length-1, ragged); tags cycle text/video/audio."""
    parts = []
    for i, n in enumerate(lengths):
        tg = (tags[i] if tags is not None else (TAG_TEXT, TAG_VIDEO, TAG_AUDIO)[i % 3])
        p = _video_positions(n, 4, 5) if tg == TAG_VIDEO else _text_positions(n)
        parts.append((["text", "video", "audio"][tg], int(n), p, tg))
    N = int(sum(lengths))
    return _assemble(f"random_{seed}", seed, heads, head_dim, parts, [0, N], [0.0], capacity, scale)


def video_segment_16k(seed: int = 6) -> PackedWorkload:
    """One 16,384-token video segment (4 latent frames of 64x64), 40 x 128: a smaller case of the
    H3 attention shape for profiling (each of Q, K, V, O is 168 MB, larger than the 129 MB L2)."""
    parts = [("video", 16384, _video_positions(16384, 64, 64), TAG_VIDEO)]
    return _assemble("video_segment_16384tok_40x128", seed, 40, 128, parts, [0, 16384], [0.0], None)


@dataclass
class VsaWorkload:
    """A 3D latent grid (T, H, W) in row-major token order, attended over selected blocks."""

    name: str
    num_heads: int
    head_dim: int
    grid: Tuple[int, int, int]
    block: Tuple[int, int, int]
    topk: int
    q: torch.Tensor  # bf16 [N, H, D]
    k: torch.Tensor
    v: torch.Tensor

    @property
    def num_tokens(self) -> int:
        t, h, w = self.grid
        return t * h * w


def vsa_video(seed: int = 7, grid=(32, 48, 84), block=(4, 4, 4), heads: int = 24,
              head_dim: int = 128, topk: Optional[int] = None) -> VsaWorkload:
    """Q/K/V ~ N(0,1) in bf16 over a (T, H, W) latent grid; 32x48x84 is the latent of a
    1344x768 video (16x spatial compression), the resolution the pages quote for VSA.  topk
    defaults to 1/8 of the blocks (rounded down, at least 1)."""
    rng = np.random.default_rng(seed)
    n = grid[0] * grid[1] * grid[2]
    nblk = 1
    for L, b in zip(grid, block):
        nblk *= (L + b - 1) // b
    k_sel = max(1, nblk // 8) if topk is None else int(topk)
    q, k, v = (_normal_bf16(rng, (n, heads, head_dim)) for _ in range(3))
    return VsaWorkload(name=f"vsa_{grid[0]}x{grid[1]}x{grid[2]}_b{block[0]}x{block[1]}x{block[2]}_top{k_sel}",
                       num_heads=heads, head_dim=head_dim, grid=tuple(grid), block=tuple(block),
                       topk=k_sel, q=q, k=k, v=v)


def vsa_paired_selection(seed: int, heads: int, nblk: int, topk: int, shared: int) -> np.ndarray:
    """A block selection int32 [heads, nblk, topk] (ascending ids, distinct per list) in which
    query blocks 2p and 2p + 1 have exactly `shared` selected blocks in common and the rest drawn
    at random from the other blocks: a stand-in for the overlap of neighbouring query blocks'
    selections on spatially coherent latents (random N(0,1) inputs give about topk^2 / nblk)."""
    rng = np.random.default_rng(seed)
    sel = np.empty((heads, nblk, topk), np.int32)
    for h in range(heads):
        for p in range(0, nblk, 2):
            a = rng.choice(nblk, topk, replace=False)
            rest = np.setdiff1d(np.arange(nblk), a)
            b = np.concatenate([a[:shared], rng.choice(rest, topk - shared, replace=False)])
            sel[h, p] = np.sort(a)
            if p + 1 < nblk:
                sel[h, p + 1] = np.sort(b)
    return sel


WORKLOADS = {
    "tiny_example": tiny_example,
    "single_request_4k": single_request_4k,
    "h3_full_request": h3_full_request,
    "continuation_batch": continuation_batch,
    "continuation_batch_4seg": lambda: continuation_batch(per_request_segments=True),
    "window_grid": window_grid,
    "video_segment_16k": video_segment_16k,
    "vsa_video": vsa_video,
}
