"""Host-side checks of the C ABI (no GPU): the library loads, exports every symbol the header
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "h3attn.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import packed_varlen_attention_modality_gb300 as h3

    return h3.load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"H3_API\s+[\w\s\*]+?\b(h3_\w+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = _declared()
    for must in ["h3_rope_apply", "h3_varlen_attn_fwd", "h3_varlen_attn_workspace_size",
                 "h3_window_count", "h3_window_pack", "h3_window_unpack", "h3_get_device_error",
                 "h3_status_string", "h3_version"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    import subprocess
    import packed_varlen_attention_modality_gb300 as h3

    out = subprocess.run(["nm", "-D", "--defined-only", h3.lib_path()], capture_output=True, text=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if " T " in l})
    assert exported == _declared()


def test_workspace_size_grows_with_segments(lib):
    sizes = [lib.h3_varlen_attn_workspace_size(s, 40, 58000, 128) for s in (1, 3, 693, 65535)]
    assert all(x % 256 == 0 for x in sizes) and sizes == sorted(sizes)
    assert sizes[-1] >= 8 * 65535 and lib.h3_varlen_attn_workspace_size(0, 40, 1, 128) == 0


def test_wait_limit_setting_returns_the_previous_and_zero_restores_the_default(lib):
    default = 2_000_000_000
    assert lib.h3_set_wait_limit_ns(0) == default
    assert lib.h3_set_wait_limit_ns(1500) == default
    assert lib.h3_set_wait_limit_ns(0) == 1500
    assert lib.h3_set_wait_limit_ns(0) == default


def test_stall_setting_returns_the_previous(lib):
    assert lib.h3_debug_stall_loads(-1) == -1
    assert lib.h3_debug_stall_loads(3) == -1
    assert lib.h3_debug_stall_loads(-5) == 3
    assert lib.h3_debug_stall_loads(-1) == -1


def test_version_and_status_strings(lib):
    assert lib.h3_version() == 100
    for s in range(11):
        assert len(lib.h3_status_string(s)) >= 2
    assert lib.h3_status_string(99) == b"unknown status"


def _i3(v):
    return (ctypes.c_int32 * 3)(*v)


@pytest.mark.parametrize("grid,win,shift", [((32, 48, 84), (4, 8, 8), (0, 0, 0)),
                                            ((32, 48, 84), (4, 8, 8), (2, 4, 4)),
                                            ((5, 6, 7), (2, 4, 4), (1, 2, 2)),
                                            ((1, 1, 1), (4, 8, 8), (3, 7, 7))])
def test_window_count_matches_oracle(lib, grid, win, shift):
    assert lib.h3_window_count(_i3(grid), _i3(win), _i3(shift)) == oracle.window_count(grid, win, shift)


@pytest.mark.parametrize("grid,win,shift", [((0, 4, 4), (2, 2, 2), (0, 0, 0)), ((4, 4, 4), (2, 0, 2), (0, 0, 0)),
                                            ((4, 4, 4), (2, 2, 2), (2, 0, 0)), ((4, 4, 4), (2, 2, 2), (-1, 0, 0))])
def test_window_count_rejects_bad_geometry(lib, grid, win, shift):
    assert lib.h3_window_count(_i3(grid), _i3(win), _i3(shift)) == -1


FAKE = 0x1000  # never dereferenced: every call below is rejected by host-side validation


def test_attn_rejects_bad_arguments_on_the_host(lib):
    f = lib.h3_varlen_attn_fwd
    P = ctypes.c_void_p
    need = lib.h3_varlen_attn_workspace_size(3, 2, 128, 128)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cu=FAKE, S=3, maxs=128, C=256, H=2, D=128,
              ws=FAKE, wsb=need)

    def call(**kw):
        a = dict(ok, **kw)
        return f(P(a["q"]), P(a["k"]), P(a["v"]), P(a["o"]), P(a["lse"]) if a["lse"] else None,
                 P(a["cu"]) if a["cu"] else None, a["S"], a["maxs"], a["C"], a["H"], a["D"], 0.0,
                 P(a["ws"]) if a["ws"] else None, a["wsb"], None)

    assert call(q=0) == 1 and call(cu=0) == 1 and call(o=0) == 1          # H3_ERR_NULL
    assert call(S=-1) == 2 and call(H=0) == 2 and call(maxs=512) == 2      # max_seqlen > capacity
    assert call(D=96) == 4                                                # H3_ERR_UNSUPPORTED
    assert call(q=FAKE + 8) == 8 and call(lse=FAKE + 2) == 8              # H3_ERR_MISALIGNED
    assert call(ws=0) == 5 and call(wsb=need - 1) == 5                    # H3_ERR_WORKSPACE
    assert call(ws=FAKE + 4) == 8
    assert call(S=0, ws=0, wsb=0) == 0 and call(maxs=0) == 0              # nothing to do


def test_rope_rejects_bad_arguments_on_the_host(lib):
    f = lib.h3_rope_apply
    P = ctypes.c_void_p

    def call(q=FAKE, qo=FAKE, k=FAKE, ko=FAKE, n=10, H=2, D=64, pos=FAKE, tag=FAKE, cu=None, R=0, cfg=None):
        return f(P(q) if q else None, P(qo) if qo else None, P(k) if k else None, P(ko) if ko else None,
                 n, H, D, P(pos) if pos else None, P(tag) if tag else None, P(cu) if cu else None, R, None,
                 cfg, None)

    assert call(q=0) == 1 and call(pos=0) == 1 and call(ko=0) == 1
    assert call(n=-1) == 2 and call(H=0) == 2 and call(cu=FAKE, R=0) == 2
    assert call(D=80) == 4
    assert call(q=FAKE + 4) == 8
    import packed_varlen_attention_modality_gb300 as h3

    bad = h3.RopeConfig(video_dims_t=30, video_dims_h=16, video_dims_w=16)  # sums to 62 != 64
    assert call(cfg=ctypes.byref(bad)) == 2
    odd = h3.RopeConfig(video_dims_t=31, video_dims_h=17, video_dims_w=16)  # odd band width
    assert call(cfg=ctypes.byref(odd)) == 2


def test_window_calls_reject_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    src = (P * 1)(FAKE)
    dst = (P * 1)(FAKE)
    g, w, s = _i3((4, 8, 8)), _i3((2, 4, 4)), _i3((1, 2, 2))
    assert lib.h3_window_pack(g, w, s, None, P(FAKE), src, dst, 1, 256, None) == 1
    assert lib.h3_window_pack(g, w, s, P(FAKE), P(FAKE), src, dst, 9, 256, None) == 2
    assert lib.h3_window_pack(g, w, s, P(FAKE), P(FAKE), src, dst, 1, 200, None) == 8
    assert lib.h3_window_pack(g, w, _i3((2, 2, 2)), P(FAKE), P(FAKE), src, dst, 1, 256, None) == 2
    assert lib.h3_window_unpack(P(FAKE), 16, P(FAKE + 8), P(FAKE), 256, None) == 8
    assert lib.h3_window_unpack(None, 16, P(FAKE), P(FAKE), 256, None) == 1
    assert lib.h3_window_unpack(P(FAKE), -2, P(FAKE), P(FAKE), 256, None) == 2


def test_window_attention_rejects_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    f = lib.h3_window_attn_fwd
    g, w, sh = _i3((4, 8, 8)), _i3((4, 8, 8)), _i3((2, 4, 4))

    def call(q=FAKE, win=w, H=2, D=128, grid=g, shift=sh):
        return f(P(q) if q else None, P(FAKE), P(FAKE), P(FAKE), None, grid, win, shift, H, D, 0.0, None)

    assert call(q=0) == 1
    assert call(H=0) == 2 and call(shift=_i3((4, 0, 0))) == 2
    assert call(D=96) == 4
    assert call(win=_i3((4, 8, 12))) == 4   # 8*12 does not divide 128
    assert call(win=_i3((8, 8, 8))) == 4    # 512 rows: more than two 128-row tiles
    assert call(q=FAKE + 8) == 8


@pytest.mark.parametrize("grid,block", [((29, 40, 50), (4, 4, 4)), ((32, 48, 84), (4, 4, 4)),
                                        ((5, 9, 11), (2, 4, 8)), ((1, 1, 1), (4, 4, 4))])
def test_vsa_block_count_matches_oracle(lib, grid, block):
    assert lib.h3_vsa_block_count(_i3(grid), _i3(block)) == oracle.vsa_block_count(grid, block)
    assert lib.h3_vsa_block_count(_i3((0, 4, 4)), _i3(block)) == -1


def test_vsa_workspace_size_holds_both_block_means(lib):
    ws = lib.h3_vsa_select_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 4)), 24, 128)
    assert ws % 256 == 0 and ws >= 2 * 24 * 2016 * 128 * 4
    assert lib.h3_vsa_select_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 8)), 24, 128) == 0  # 128-token block
    assert lib.h3_vsa_select_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 4)), 24, 96) == 0


def test_vsa_calls_reject_bad_arguments_on_the_host(lib):
    P = ctypes.c_void_p
    g, b = _i3((8, 8, 8)), _i3((4, 4, 4))   # 8 blocks
    ws = lib.h3_vsa_select_workspace_size(g, b, 2, 128)

    def sel(q=FAKE, topk=3, D=128, block=b, wsb=ws, w=FAKE, scores=FAKE):
        return lib.h3_vsa_select(P(q) if q else None, P(FAKE), g, block, 2, D, topk, 0.0,
                                 P(scores) if scores else None, P(FAKE), P(w) if w else None, wsb, None)

    assert sel(q=0) == 1 and sel(scores=0) == 1
    assert sel(topk=0) == 2 and sel(topk=9) == 2
    assert sel(D=96) == 4 and sel(block=_i3((4, 4, 8))) == 4
    assert sel(w=0) == 5 and sel(wsb=ws - 1) == 5
    assert sel(q=FAKE + 8) == 8 and sel(scores=FAKE + 2) == 8

    aws = lib.h3_vsa_attn_workspace_size(g, b, 2, 3)
    assert aws > 0 and lib.h3_vsa_attn_workspace_size(g, b, 2, 9) == 0

    def attn(q=FAKE, topk=3, D=128, block=b, idx=FAKE, w=FAKE, wsb=aws):
        return lib.h3_vsa_attn_fwd(P(q) if q else None, P(FAKE), P(FAKE), P(FAKE), None, g, block, 2, D,
                                   P(idx) if idx else None, topk, 0.0, P(w) if w else None, wsb, None)

    assert attn(q=0) == 1 and attn(idx=0) == 1
    assert attn(topk=0) == 2 and attn(topk=9) == 2
    assert attn(D=64, block=_i3((2, 2, 2))) == 4
    assert attn(w=0) == 5 and attn(wsb=aws - 1) == 5
    assert attn(q=FAKE + 8) == 8 and attn(idx=FAKE + 2) == 8 and attn(w=FAKE + 8) == 8


def test_vsa_attn_workspace_holds_the_schedule(lib):
    # 2016 blocks -> 1008 pairs per head; 8 bytes per step, topk steps per pair, plus a count per pair
    ws = lib.h3_vsa_attn_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 4)), 24, 252)
    assert ws >= 24 * 1008 * (252 * 8 + 4)
    assert lib.h3_vsa_attn_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 4)), 24, 2017) == 0
    assert lib.h3_vsa_attn_workspace_size(_i3((32, 48, 84)), _i3((4, 4, 8)), 24, 1) == 0


def _plan_fields(p):
    return (p.tail_start, p.start_frame, p.audio_cut, tuple(p.group_rows), tuple(p.group_offset),
            p.num_rows, p.keep_video_from, p.keep_audio_from, p.out_video_frames, p.out_audio_rows)


def test_continuation_plan_matches_oracle_on_random_windows(lib):
    import packed_varlen_attention_modality_gb300 as h3

    rng = np.random.default_rng(21)
    cases = [(558, 29, 200, 40, 50, 29, 200, 7, 4), (5, 245, 500, 2, 3, 20, 150, 7, 1),
             (0, 7, 0, 1, 1, 7, 0, 7, 4), (3, 40, 9, 2, 2, 9, 30, 7, 4)]
    for _ in range(200):
        tail = int(rng.integers(0, 9))
        clip_f = tail + int(rng.integers(0, 40))
        fpl = int(rng.integers(1, 6))
        clip_a = int(rng.integers(0, 400))
        cut = min(((clip_f - tail) * fpl * 40) // 24, clip_a)
        cases.append((int(rng.integers(0, 600)), clip_f, clip_a, int(rng.integers(1, 9)),
                      int(rng.integers(1, 9)), tail + int(rng.integers(0, 40)),
                      (clip_a - cut) + int(rng.integers(0, 300)), tail, fpl))
    for c in cases:
        ref = oracle.continuation_plan(*c[:7], tail_frames=c[7], frames_per_latent=c[8])
        got = h3.continuation_plan(h3.continuation_config(*c))
        assert _plan_fields(got) == (ref.tail_start, ref.start_frame, ref.audio_cut, ref.group_rows,
                                     ref.group_offset, ref.num_rows, ref.keep_video_from,
                                     ref.keep_audio_from, ref.out_video_frames, ref.out_audio_rows), c


def test_continuation_calls_reject_bad_arguments_on_the_host(lib):
    import packed_varlen_attention_modality_gb300 as h3

    P = ctypes.c_void_p
    bad = [h3.continuation_config(5, 6, 40, 2, 2, 10, 40),      # clip shorter than the tail
           h3.continuation_config(5, 10, 40, 2, 2, 6, 40),      # new window shorter than the tail
           h3.continuation_config(5, 29, 200, 2, 2, 29, 10),    # new audio shorter than the audio tail
           h3.continuation_config(-1, 29, 200, 2, 2, 29, 200), h3.continuation_config(5, 29, 200, 0, 2, 29, 200)]
    plan = h3.ContinuationPlan()
    for c in bad:
        assert lib.h3_continuation_make_plan(ctypes.byref(c), ctypes.byref(plan)) == 2
    assert lib.h3_continuation_make_plan(None, ctypes.byref(plan)) == 1
    good = h3.continuation_config(5, 29, 200, 2, 2, 29, 200)
    f = lib.h3_continuation_pack

    def pack(rb=64, rows=FAKE, text=FAKE):
        return f(ctypes.byref(good), P(text) if text else None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), rb,
                 P(rows) if rows else None, P(FAKE), P(FAKE), P(FAKE), None)

    assert pack(rows=0) == 1 and pack(text=0) == 1
    assert pack(rb=24) == 2 and pack(rb=0) == 2
    assert pack(rows=FAKE + 8) == 8
    g = lib.h3_continuation_append
    assert g(ctypes.byref(good), P(FAKE), P(FAKE), 64, P(FAKE), 10, P(FAKE), 10**6, None) == 2  # video capacity
    assert g(ctypes.byref(good), P(FAKE), P(FAKE), 64, P(FAKE), 10**6, P(FAKE), 10, None) == 2  # audio capacity
    assert g(ctypes.byref(good), None, P(FAKE), 64, P(FAKE), 10**6, P(FAKE), 10**6, None) == 1
    m = lib.h3_masked_row_update
    assert m(P(FAKE), P(FAKE), P(FAKE), 4, 24, None) == 2 and m(None, P(FAKE), P(FAKE), 4, 32, None) == 1
    assert m(P(FAKE + 8), P(FAKE), P(FAKE), 4, 32, None) == 8 and m(None, None, None, 0, 32, None) == 0
