"""GB300-native packed varlen attention with modality-tagged 3D RoPE.

Thin Python binding over the C ABI of ``libh3attn.so`` (declared in include/h3attn.h).  It only
marshals arguments -- checks dtypes and shapes, takes device pointers and the current CUDA
stream from PyTorch tensors -- and every step of the computation runs in the library's CUDA
kernels.  There is no CPU or PyTorch fallback: if the library is missing, every call raises.

Calls:
  rope_apply        modality-tagged RoPE of Q and K with the continuation time shift
  varlen_attn_fwd   block-diagonal softmax attention over cu_seqlens segments
  window_count / window_pack / window_unpack   shifted 3D window partition and row gather/scatter
  window_attn_fwd   shifted 3D window attention read and written in place on the grid
  vsa_select / vsa_attn_fwd   block-sparse video attention: block gate scores + top-k
                    selection, then attention over the selected 64-token blocks (paired query
                    blocks share the key blocks both selected)
  continuation_plan / continuation_pack / continuation_append / masked_row_update
                    continuation window: tails, five row groups, overlap discard, target updates
  sp_assign_windows / sp_rank_tokens / sp_layer_order / sp_exchange_plan
                    window-aligned sequence parallelism: window owners, local orders and the
                    all-to-all plan of a regular <-> shifted switch (host planning; the caller
                    moves the rows with its own all-to-all)
  get_device_error  read (and clear) the device-side error word
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

__all__ = ["H3Error", "RopeConfig", "lib_path", "load_library", "rope_apply", "varlen_attn_fwd",
           "varlen_attn_fwd_noalloc", "window_attn_fwd", "vsa_block_count",
           "vsa_select_workspace_size", "vsa_select", "vsa_attn_workspace_size", "vsa_attn_fwd",
           "ContinuationConfig",
           "ContinuationPlan", "continuation_config", "continuation_plan", "continuation_pack",
           "continuation_append", "masked_row_update", "sp_assign_windows", "sp_layer_order",
           "sp_rank_tokens", "sp_exchange_plan",
           "varlen_attn_workspace_size", "window_count", "window_pack", "window_unpack",
           "get_device_error", "TAG_TEXT", "TAG_VIDEO", "TAG_AUDIO"]

TAG_TEXT, TAG_VIDEO, TAG_AUDIO = 0, 1, 2

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libh3attn.so"
_lib = None

_STATUS = {0: "H3_OK", 1: "H3_ERR_NULL", 2: "H3_ERR_INVALID_ARG", 3: "H3_ERR_BAD_CU_SEQLENS",
           4: "H3_ERR_UNSUPPORTED", 5: "H3_ERR_WORKSPACE", 6: "H3_ERR_CUDA", 7: "H3_ERR_TIMEOUT",
           8: "H3_ERR_MISALIGNED", 9: "H3_ERR_BAD_PERM", 10: "H3_ERR_BAD_BLOCK_INDEX"}


class H3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.name = _STATUS.get(self.status, f"status {status}")
        msg = load_library().h3_status_string(self.status).decode()
        super().__init__(f"{where}: {self.name}: {msg}")


class RopeConfig(ctypes.Structure):
    """Mirror of h3_rope_cfg; zero fields select the defaults (base 10000, D/2:D/4:D/4, 40/24)."""
    _fields_ = [("base_text", ctypes.c_float), ("base_video", ctypes.c_float),
                ("base_audio", ctypes.c_float), ("video_dims_t", ctypes.c_int32),
                ("video_dims_h", ctypes.c_int32), ("video_dims_w", ctypes.c_int32),
                ("audio_hz", ctypes.c_float), ("video_fps", ctypes.c_float)]


_I = ctypes.c_int32


class ContinuationConfig(ctypes.Structure):
    """Mirror of h3_continuation_cfg."""
    _fields_ = [("text_rows", _I), ("clip_video_frames", _I), ("clip_audio_rows", _I),
                ("frame_h", _I), ("frame_w", _I), ("new_video_frames", _I), ("new_audio_rows", _I),
                ("tail_frames", _I), ("frames_per_latent", _I)]


class ContinuationPlan(ctypes.Structure):
    """Mirror of h3_continuation_plan."""
    _fields_ = [("tail_start", _I), ("start_frame", _I), ("audio_cut", _I), ("group_rows", _I * 5),
                ("group_offset", _I * 6), ("num_rows", _I), ("keep_video_from", _I),
                ("keep_audio_from", _I), ("out_video_frames", _I), ("out_audio_rows", _I)]


def lib_path() -> str:
    return os.path.join(_PKG_DIR, _LIB_NAME)


def load_library():
    """Load libh3attn.so (built in-tree by __graft_entry__.build()); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; "
                           "g.build()'` first (this package has no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, I32, U64, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    I32P = ctypes.POINTER(ctypes.c_int32)
    sigs = {
        "h3_rope_apply": (I32, [P, P, P, P, I32, I32, I32, P, P, P, I32, P,
                                ctypes.POINTER(RopeConfig), P]),
        "h3_varlen_attn_workspace_size": (U64, [I32, I32, I32, I32]),
        "h3_varlen_attn_fwd": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, F32, P, U64, P]),
        "h3_varlen_attn_fwd_noalloc": (I32, [P, P, P, P, P, P, I32, I32, I32, I32, I32, F32, P]),
        "h3_window_attn_fwd": (I32, [P, P, P, P, P, I32P, I32P, I32P, I32, I32, F32, P]),
        "h3_window_count": (I32, [I32P, I32P, I32P]),
        "h3_window_pack": (I32, [I32P, I32P, I32P, P, P, ctypes.POINTER(P), ctypes.POINTER(P),
                                 I32, I32, P]),
        "h3_window_unpack": (I32, [P, I32, P, P, I32, P]),
        "h3_vsa_block_count": (I32, [I32P, I32P]),
        "h3_continuation_make_plan": (I32, [ctypes.POINTER(ContinuationConfig), ctypes.POINTER(ContinuationPlan)]),
        "h3_continuation_pack": (I32, [ctypes.POINTER(ContinuationConfig), P, P, P, P, P, I32, P, P, P, P, P]),
        "h3_continuation_append": (I32, [ctypes.POINTER(ContinuationConfig), P, P, I32, P, ctypes.c_int64, P,
                                         ctypes.c_int64, P]),
        "h3_masked_row_update": (I32, [P, P, P, I32, I32, P]),
        "h3_sp_assign_windows": (I32, [I32P, I32P, I32P, I32, P, P]),
        "h3_sp_rank_tokens": (I32, [I32P, I32P, I32P, P, I32, P]),
        "h3_sp_layer_order": (I32, [I32P, I32P, I32P, P, I32, I32, P, ctypes.c_int64]),
        "h3_sp_exchange_plan": (I32, [I32P, I32P, I32P, P, I32P, P, I32, I32, P, P, P, P]),
        "h3_vsa_select_workspace_size": (U64, [I32P, I32P, I32, I32]),
        "h3_vsa_select": (I32, [P, P, I32P, I32P, I32, I32, I32, F32, P, P, P, U64, P]),
        "h3_vsa_attn_workspace_size": (U64, [I32P, I32P, I32, I32]),
        "h3_vsa_attn_fwd": (I32, [P, P, P, P, P, I32P, I32P, I32, I32, P, I32, F32, P, U64, P]),
        "h3_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
        "h3_debug_stall_loads": (I32, [I32]),
        "h3_get_device_error": (I32, [P]),
        "h3_status_string": (ctypes.c_char_p, [I32]),
        "h3_version": (I32, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise H3Error(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _require(t: torch.Tensor, name: str, dtype, device: torch.device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _i3(v: Sequence[int]):
    a = (ctypes.c_int32 * 3)(*[int(x) for x in v])
    return a


def rope_apply(q: torch.Tensor, k: Optional[torch.Tensor], pos: torch.Tensor, tag: torch.Tensor,
               cu_requests: Optional[torch.Tensor] = None, start_frames: Optional[torch.Tensor] = None,
               num_tokens: Optional[int] = None, q_out: Optional[torch.Tensor] = None,
               k_out: Optional[torch.Tensor] = None, cfg: Optional[RopeConfig] = None):
    """Tagged RoPE of q (and k) [C, H, D] bf16; in place unless q_out / k_out are given.

    pos fp32 [>=N, 3] (t, h, w); tag uint8 [>=N]; cu_requests int32 [R+1] and start_frames fp32
    [R] (continuation start frames s_r) are optional.  Returns (q_out, k_out).
    """
    dev = q.device
    _require(q, "q", torch.bfloat16, dev)
    if q.dim() != 3:
        raise ValueError("q must be [C, H, D]")
    C, H, D = q.shape
    n = C if num_tokens is None else int(num_tokens)
    if n > C:
        raise ValueError("num_tokens exceeds the capacity of q")
    q_out = q if q_out is None else q_out
    _require(q_out, "q_out", torch.bfloat16, dev)
    if k is not None:
        _require(k, "k", torch.bfloat16, dev)
        k_out = k if k_out is None else k_out
        _require(k_out, "k_out", torch.bfloat16, dev)
        if k.shape != q.shape or k_out.shape != q.shape:
            raise ValueError("k must have q's shape")
    else:
        k_out = None
    if q_out.shape != q.shape:
        raise ValueError("q_out must have q's shape")
    _require(pos, "pos", torch.float32, dev)
    _require(tag, "tag", torch.uint8, dev)
    if pos.shape[0] < n or tag.shape[0] < n:
        raise ValueError("pos / tag must cover num_tokens rows")
    nreq = 0
    if cu_requests is not None:
        _require(cu_requests, "cu_requests", torch.int32, dev)
        nreq = cu_requests.numel() - 1
    if start_frames is not None:
        _require(start_frames, "start_frames", torch.float32, dev)
        if cu_requests is not None and start_frames.numel() < nreq:
            raise ValueError("start_frames must have one entry per request")
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_rope_apply(_ptr(q), _ptr(q_out), _ptr(k), _ptr(k_out), n, H, D, _ptr(pos),
                               _ptr(tag), _ptr(cu_requests), nreq, _ptr(start_frames),
                               ctypes.byref(cfg) if cfg is not None else None, _stream(dev))
    _check(st, "h3_rope_apply")
    return q_out, k_out


def varlen_attn_workspace_size(num_segments: int, num_heads: int, max_seqlen: int, head_dim: int) -> int:
    return int(load_library().h3_varlen_attn_workspace_size(num_segments, num_heads, max_seqlen, head_dim))


def varlen_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                    max_seqlen: int, out: Optional[torch.Tensor] = None, return_lse: bool = False,
                    lse: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                    workspace: Optional[torch.Tensor] = None):
    """Block-diagonal attention over the segments of cu_seqlens (int32 [S+1], device).

    q, k, v: bf16 [C, H, D] with C >= cu_seqlens[-1].  Rows of `out` outside every segment are
    left untouched.  Returns out (and lse fp32 [H, C] when requested).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, torch.bfloat16, dev)
    if q.dim() != 3 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [C, H, D]")
    C, H, D = q.shape
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    S = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", torch.bfloat16, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if return_lse and lse is None:
        lse = torch.empty((H, C), dtype=torch.float32, device=dev)
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if tuple(lse.shape) != (H, C):
            raise ValueError("lse must be [H, C]")
    lib = load_library()
    ws_need = int(lib.h3_varlen_attn_workspace_size(S, H, int(max_seqlen), D))
    if ws_need > 0 and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    with torch.cuda.device(dev):
        st = lib.h3_varlen_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                    _ptr(cu_seqlens), S, int(max_seqlen), C, H, D, scale,
                                    _ptr(workspace), ws_bytes, _stream(dev))
    _check(st, "h3_varlen_attn_fwd")
    return (out, lse) if (return_lse or lse is not None) else out


def varlen_attn_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            cu_seqlens: torch.Tensor, max_seqlen: int, out: torch.Tensor,
                            lse: Optional[torch.Tensor] = None,
                            softmax_scale: Optional[float] = None) -> torch.Tensor:
    """varlen_attn_fwd through the entry point that allocates no device memory.

    For callers that cannot allocate: `out` (and `lse`, if wanted) must be given, and the
    library uses its own fixed scratch array (at most 16384 segments).  Calls on one device must
    not overlap on the GPU; the first call on a device should come before any stream capture.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _require(t, name, torch.bfloat16, dev)
    if q.dim() != 3 or k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
        raise ValueError("q, k, v, out must all be [C, H, D]")
    C, H, D = q.shape
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if tuple(lse.shape) != (H, C):
            raise ValueError("lse must be [H, C]")
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_varlen_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                            _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                            int(max_seqlen), C, H, D, scale, _stream(dev))
    _check(st, "h3_varlen_attn_fwd_noalloc")
    return out


def window_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, grid: Sequence[int],
                    win: Sequence[int], shift: Sequence[int], out: Optional[torch.Tensor] = None,
                    return_lse: bool = False, lse: Optional[torch.Tensor] = None,
                    softmax_scale: Optional[float] = None):
    """Shifted 3D window attention in place on the grid (no packed copies).

    q, k, v: bf16 [T*H*W, heads, D] in row-major (t, h, w) token order.  Returns out (and lse
    fp32 [heads, T*H*W] when requested), in the same order.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, torch.bfloat16, dev)
    n = int(grid[0]) * int(grid[1]) * int(grid[2])
    if q.dim() != 3 or q.shape[0] != n or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [T*H*W, heads, D]")
    _, H, D = q.shape
    out = torch.empty_like(q) if out is None else out
    _require(out, "out", torch.bfloat16, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if return_lse and lse is None:
        lse = torch.empty((H, n), dtype=torch.float32, device=dev)
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if tuple(lse.shape) != (H, n):
            raise ValueError("lse must be [heads, T*H*W]")
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_window_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _i3(grid),
                                    _i3(win), _i3(shift), H, D, scale, _stream(dev))
    _check(st, "h3_window_attn_fwd")
    return (out, lse) if (return_lse or lse is not None) else out


def window_count(grid: Sequence[int], win: Sequence[int], shift: Sequence[int]) -> int:
    n = load_library().h3_window_count(_i3(grid), _i3(win), _i3(shift))
    if n < 0:
        raise ValueError("invalid window geometry")
    return int(n)


def window_pack(grid: Sequence[int], win: Sequence[int], shift: Sequence[int],
                tensors: Sequence[torch.Tensor] = (), device: Optional[torch.device] = None,
                perm: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                outs: Optional[Sequence[torch.Tensor]] = None):
    """Partition the (T, H, W) grid into (shifted) windows and gather each tensor's rows.

    tensors: [N, ...] contiguous, same device, N = T*H*W.  Returns (perm, cu_seqlens, packed).
    """
    nwin = window_count(grid, win, shift)
    n = int(grid[0]) * int(grid[1]) * int(grid[2])
    dev = tensors[0].device if tensors else (device or torch.device("cuda"))
    if perm is None:
        perm = torch.empty(n, dtype=torch.int32, device=dev)
    if cu_seqlens is None:
        cu_seqlens = torch.empty(nwin + 1, dtype=torch.int32, device=dev)
    _require(perm, "perm", torch.int32, dev)
    _require(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if perm.numel() < n or cu_seqlens.numel() < nwin + 1:
        raise ValueError("perm / cu_seqlens too small")
    outs = list(outs) if outs is not None else [torch.empty_like(t) for t in tensors]
    row_bytes = 0
    for i, (t, o) in enumerate(zip(tensors, outs)):
        if not t.is_contiguous() or not o.is_contiguous() or t.device != dev or o.device != dev:
            raise ValueError("window_pack tensors must be contiguous on one device")
        if t.shape[0] != n or o.shape != t.shape or o.dtype != t.dtype:
            raise ValueError("each tensor must have T*H*W rows and a matching output")
        rb = t[0].numel() * t.element_size()
        if i and rb != row_bytes:
            raise ValueError("all tensors must share one row size")
        row_bytes = rb
    k = len(tensors)
    src = (ctypes.c_void_p * max(k, 1))(*[t.data_ptr() for t in tensors])
    dst = (ctypes.c_void_p * max(k, 1))(*[o.data_ptr() for o in outs])
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_window_pack(_i3(grid), _i3(win), _i3(shift), _ptr(perm), _ptr(cu_seqlens),
                                src, dst, k, row_bytes, _stream(dev))
    _check(st, "h3_window_pack")
    return perm, cu_seqlens, outs


def window_unpack(perm: torch.Tensor, src: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Restore original order: out[perm[j]] = src[j]."""
    dev = src.device
    _require(perm, "perm", torch.int32, dev)
    if not src.is_contiguous():
        raise ValueError("src must be contiguous")
    n = src.shape[0]
    if perm.numel() < n:
        raise ValueError("perm too small")
    out = torch.empty_like(src) if out is None else out
    if out.shape != src.shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError("out must match src")
    row_bytes = src[0].numel() * src.element_size()
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_window_unpack(_ptr(perm), n, _ptr(src), _ptr(out), row_bytes, _stream(dev))
    _check(st, "h3_window_unpack")
    return out


def vsa_block_count(grid: Sequence[int], block: Sequence[int] = (4, 4, 4)) -> int:
    n = load_library().h3_vsa_block_count(_i3(grid), _i3(block))
    if n < 0:
        raise ValueError("invalid VSA block geometry")
    return int(n)


def vsa_select_workspace_size(grid: Sequence[int], block: Sequence[int], num_heads: int,
                              head_dim: int) -> int:
    return int(load_library().h3_vsa_select_workspace_size(_i3(grid), _i3(block), num_heads, head_dim))


def vsa_select(q: torch.Tensor, k: torch.Tensor, grid: Sequence[int], topk: int,
               block: Sequence[int] = (4, 4, 4), scores: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               softmax_scale: Optional[float] = None):
    """Block gate scores and top-k key blocks per query block (VSA).

    q, k: bf16 [T*H*W, heads, D] in row-major (t, h, w) order.  Returns (block_idx int32
    [heads, nblk, topk] in ascending block id, scores fp32 [heads, nblk, nblk]).
    """
    dev = q.device
    _require(q, "q", torch.bfloat16, dev)
    _require(k, "k", torch.bfloat16, dev)
    n = int(grid[0]) * int(grid[1]) * int(grid[2])
    if q.dim() != 3 or q.shape[0] != n or k.shape != q.shape:
        raise ValueError("q, k must be [T*H*W, heads, D]")
    _, H, D = q.shape
    nblk = vsa_block_count(grid, block)
    if scores is None:
        scores = torch.empty((H, nblk, nblk), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((H, nblk, int(topk)), dtype=torch.int32, device=dev)
    _require(scores, "scores", torch.float32, dev)
    _require(out, "out", torch.int32, dev)
    if tuple(scores.shape) != (H, nblk, nblk) or tuple(out.shape) != (H, nblk, int(topk)):
        raise ValueError("scores must be [heads, nblk, nblk] and out [heads, nblk, topk]")
    need = vsa_select_workspace_size(grid, block, H, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", torch.uint8, dev)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_vsa_select(_ptr(q), _ptr(k), _i3(grid), _i3(block), H, D, int(topk), scale,
                               _ptr(scores), _ptr(out), _ptr(workspace), workspace.numel(),
                               _stream(dev))
    _check(st, "h3_vsa_select")
    return out, scores


def vsa_attn_workspace_size(grid: Sequence[int], block: Sequence[int], num_heads: int,
                            topk: int) -> int:
    return int(load_library().h3_vsa_attn_workspace_size(_i3(grid), _i3(block), num_heads, topk))


def vsa_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, grid: Sequence[int],
                 block_idx: torch.Tensor, block: Sequence[int] = (4, 4, 4),
                 out: Optional[torch.Tensor] = None, return_lse: bool = False,
                 lse: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
                 workspace: Optional[torch.Tensor] = None):
    """Token-level attention of every query block over its selected key blocks (VSA).

    q, k, v: bf16 [T*H*W, heads, D] in row-major (t, h, w) order; block_idx int32
    [heads, nblk, topk]; workspace uint8 of vsa_attn_workspace_size() bytes (allocated when
    omitted).  Returns out (and lse fp32 [heads, T*H*W] when requested).
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, torch.bfloat16, dev)
    n = int(grid[0]) * int(grid[1]) * int(grid[2])
    if q.dim() != 3 or q.shape[0] != n or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [T*H*W, heads, D]")
    _, H, D = q.shape
    nblk = vsa_block_count(grid, block)
    _require(block_idx, "block_idx", torch.int32, dev)
    if block_idx.dim() != 3 or tuple(block_idx.shape[:2]) != (H, nblk):
        raise ValueError("block_idx must be [heads, nblk, topk]")
    topk = int(block_idx.shape[2])
    out = torch.empty_like(q) if out is None else out
    _require(out, "out", torch.bfloat16, dev)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if return_lse and lse is None:
        lse = torch.empty((H, n), dtype=torch.float32, device=dev)
    if lse is not None:
        _require(lse, "lse", torch.float32, dev)
        if tuple(lse.shape) != (H, n):
            raise ValueError("lse must be [heads, T*H*W]")
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    need = vsa_attn_workspace_size(grid, block, H, topk)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", torch.uint8, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        st = lib.h3_vsa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _i3(grid),
                                 _i3(block), H, D, _ptr(block_idx), topk, scale, _ptr(workspace),
                                 workspace.numel(), _stream(dev))
    _check(st, "h3_vsa_attn_fwd")
    return (out, lse) if (return_lse or lse is not None) else out


def continuation_config(text_rows: int, clip_video_frames: int, clip_audio_rows: int, frame_h: int,
                        frame_w: int, new_video_frames: int, new_audio_rows: int, tail_frames: int = 7,
                        frames_per_latent: int = 4) -> ContinuationConfig:
    return ContinuationConfig(text_rows, clip_video_frames, clip_audio_rows, frame_h, frame_w,
                              new_video_frames, new_audio_rows, tail_frames, frames_per_latent)


def continuation_plan(cfg: ContinuationConfig) -> ContinuationPlan:
    """Index math of a continuation window (host only)."""
    plan = ContinuationPlan()
    _check(load_library().h3_continuation_make_plan(ctypes.byref(cfg), ctypes.byref(plan)),
           "h3_continuation_make_plan")
    return plan


def _rows2d(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None, 0
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t, t[0].numel() * t.element_size() if t.shape[0] > 0 else 0


def continuation_pack(cfg: ContinuationConfig, text, clip_video, clip_audio, new_video, new_audio,
                      out: Optional[torch.Tensor] = None):
    """The five-group DiT sequence of a continuation window: returns (rows, pos fp32 [N, 3],
    tag u8 [N], target u8 [N]).  Row tensors are [n, ...] with one common row size."""
    plan = continuation_plan(cfg)
    srcs = [text, clip_video, clip_audio, new_video, new_audio]
    ref = next(t for t in srcs if t is not None and t.shape[0] > 0)
    dev = ref.device
    row_bytes = ref[0].numel() * ref.element_size()
    for i, t in enumerate(srcs):
        if t is not None and t.shape[0] > 0:
            _, rb = _rows2d(t, f"source {i}")
            if rb != row_bytes or t.dtype != ref.dtype:
                raise ValueError("all row tensors need the same row size and dtype")
    n = plan.num_rows
    out = torch.empty((n,) + tuple(ref.shape[1:]), dtype=ref.dtype, device=dev) if out is None else out
    pos = torch.empty((n, 3), dtype=torch.float32, device=dev)
    tag = torch.empty(n, dtype=torch.uint8, device=dev)
    target = torch.empty(n, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = load_library().h3_continuation_pack(ctypes.byref(cfg), _ptr(text), _ptr(clip_video),
                                                 _ptr(clip_audio), _ptr(new_video), _ptr(new_audio),
                                                 row_bytes, _ptr(out), _ptr(pos), _ptr(tag), _ptr(target),
                                                 _stream(dev))
    _check(st, "h3_continuation_pack")
    return out, pos, tag, target


def continuation_append(cfg: ContinuationConfig, new_video: torch.Tensor, new_audio: torch.Tensor,
                        clip_video: torch.Tensor, clip_audio: torch.Tensor):
    """Append the new window's rows past the overlap to the clip buffers (in place; they must
    have room for the plan's out_video_frames / out_audio_rows).  Returns the plan."""
    plan = continuation_plan(cfg)
    ref = new_video if new_video.shape[0] > 0 else new_audio
    row_bytes = ref[0].numel() * ref.element_size()
    dev = ref.device
    hw = cfg.frame_h * cfg.frame_w
    with torch.cuda.device(dev):
        st = load_library().h3_continuation_append(ctypes.byref(cfg), _ptr(new_video), _ptr(new_audio),
                                                   row_bytes, _ptr(clip_video), clip_video.shape[0],
                                                   _ptr(clip_audio), clip_audio.shape[0], _stream(dev))
    _check(st, "h3_continuation_append")
    assert plan.out_video_frames * hw <= clip_video.shape[0]
    return plan


def masked_row_update(dst: torch.Tensor, src: torch.Tensor, mask: torch.Tensor) -> torch.Tensor:
    """dst[i] = src[i] where mask[i] (uint8) is non-zero; in place on dst."""
    if dst.shape != src.shape or dst.dtype != src.dtype or mask.dtype != torch.uint8:
        raise ValueError("dst and src must match; mask must be uint8")
    n = dst.shape[0]
    row_bytes = dst[0].numel() * dst.element_size() if n > 0 else 16
    with torch.cuda.device(dst.device):
        st = load_library().h3_masked_row_update(_ptr(dst), _ptr(src), _ptr(mask), n, row_bytes,
                                                 _stream(dst.device))
    _check(st, "h3_masked_row_update")
    return dst


def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None and a.size else None


def sp_assign_windows(grid: Sequence[int], win: Sequence[int], shift: Sequence[int], world: int):
    """Owner rank of every window of one layer (longest-first on token counts) and the tokens
    each rank owns: (window_rank int32 [nwin], rank_tokens int64 [world]) as numpy arrays."""
    import numpy as np

    owner = np.empty(window_count(grid, win, shift), dtype=np.int32)
    tokens = np.empty(int(world), dtype=np.int64)
    _check(load_library().h3_sp_assign_windows(_i3(grid), _i3(win), _i3(shift), int(world),
                                               _np_ptr(owner), _np_ptr(tokens)), "h3_sp_assign_windows")
    return owner, tokens


def sp_layer_order(grid, win, shift, window_rank, world: int, rank: int):
    """Original token indices a rank holds in one layer, in its local order (numpy int32)."""
    import numpy as np

    owner = np.ascontiguousarray(window_rank, dtype=np.int32)
    n = int(sp_rank_tokens(grid, win, shift, owner, world)[rank])
    order = np.empty(max(n, 1), dtype=np.int32)
    _check(load_library().h3_sp_layer_order(_i3(grid), _i3(win), _i3(shift), _np_ptr(owner), int(world),
                                            int(rank), _np_ptr(order), n), "h3_sp_layer_order")
    return order[:n]


def sp_rank_tokens(grid, win, shift, window_rank, world: int):
    """Tokens each rank owns under a given window -> rank map (numpy int64 [world])."""
    import numpy as np

    owner = np.ascontiguousarray(window_rank, dtype=np.int32)
    tokens = np.empty(int(world), dtype=np.int64)
    _check(load_library().h3_sp_rank_tokens(_i3(grid), _i3(win), _i3(shift), _np_ptr(owner), int(world),
                                            _np_ptr(tokens)), "h3_sp_rank_tokens")
    return tokens


def sp_exchange_plan(grid, win, shift_from, rank_from, shift_to, rank_to, world: int, rank: int):
    """All-to-all of a layer switch seen by one rank: dict of numpy arrays send_counts,
    send_index, recv_counts, recv_position (see h3_sp_exchange_plan)."""
    import numpy as np

    a = np.ascontiguousarray(rank_from, dtype=np.int32)
    b = np.ascontiguousarray(rank_to, dtype=np.int32)
    n_from = int(sp_rank_tokens(grid, win, shift_from, a, world)[rank])
    n_to = int(sp_rank_tokens(grid, win, shift_to, b, world)[rank])
    plan = dict(send_counts=np.empty(int(world), np.int64), send_index=np.empty(max(n_from, 1), np.int32),
                recv_counts=np.empty(int(world), np.int64), recv_position=np.empty(max(n_to, 1), np.int32))
    _check(load_library().h3_sp_exchange_plan(_i3(grid), _i3(win), _i3(shift_from), _np_ptr(a), _i3(shift_to),
                                              _np_ptr(b), int(world), int(rank),
                                              _np_ptr(plan["send_counts"]), _np_ptr(plan["send_index"]),
                                              _np_ptr(plan["recv_counts"]), _np_ptr(plan["recv_position"])),
           "h3_sp_exchange_plan")
    plan["send_index"] = plan["send_index"][:n_from]
    plan["recv_position"] = plan["recv_position"][:n_to]
    return plan


def get_device_error(device: Optional[torch.device] = None) -> int:
    """Synchronise the current stream; return and clear the device error word (0 = none)."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    lib = load_library()
    with torch.cuda.device(dev):
        return int(lib.h3_get_device_error(_stream(dev)))


def set_wait_limit_ns(nanoseconds: int) -> int:
    """Limit of the attention kernels' internal waits for later launches (0 = the 2 s default);
    returns the previous limit.  A testing hook for the timeout path: see h3_set_wait_limit_ns."""
    return int(load_library().h3_set_wait_limit_ns(int(nanoseconds)))


def debug_stall_loads(tiles: int) -> int:
    """Make each attention CTA's key/value loader stop after `tiles` tiles (negative = never);
    returns the previous setting.  A testing hook for the timeout path: see h3_debug_stall_loads."""
    return int(load_library().h3_debug_stall_loads(int(tiles)))
