"""CPU fp64 oracle for the packed varlen attention hot path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the GPU path computes.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product library never routes through it, and it shares no code, table or
helper with the CUDA sources.

Sources (page title + section):
  [H3-vLLM]  "Joint audio/video generation in production: MiniMax-H3 and vLLM-Omni"
             §3 "Packed sequence and modality identity" (modality tags choose the RoPE
             treatment; cu_seqlens restrict softmax to the own sub-sequence; the worked
             example [0,10,30] -> [0,10,30,45]);
             §6 "Boundary trim of packed attention" (only the valid length enters the kernel).
  [H3-fast]  "Breaking the engineering bottlenecks of video-generation models"
             "Crossing the time boundary", step 3 "RoPE global time alignment"
             (t_global = t_local + s*40/24, time axis only, decimals kept);
             "Breaking the memory wall: window attention across GPUs" (regular and half-shifted
             3D windows, edge windows cropped, token order restored afterwards);
             "VSA: block-sparse attention" (64-token 4x4x4 blocks, block-level gated scoring,
             top-k block selection, token-level attention between the selected blocks);
             "Crossing the time boundary", steps 1-2 and the overlap discard (7-frame video tail,
             40 Hz audio tail, five row groups, target-only updates, suffix append).

Every function here is pinned by tests/test_oracle_pins.py against closed forms, textbook
routines, brute force and the pages' printed examples.  Readings where the pages are silent
are listed in the module docstrings of ``rope`` and ``window``.
"""
from .attention import varlen_attention, attention_weights, dense_masked_attention_bruteforce
from .rope import (RopeConfig, continuation_time_shift, rope_inv_freq, rope_angles, rope_apply,
                   video_axis_split)
from .window import (axis_window_count, window_count, window_ids, window_partition,
                     window_pack, window_unpack)
from .continuation import (ContinuationPlan, continuation_plan, continuation_pack,
                           continuation_append, masked_update)
from .vsa import (vsa_block_counts, vsa_block_count, vsa_block_ids, vsa_block_means,
                  vsa_block_scores, vsa_select, vsa_attention)

__all__ = [
    "varlen_attention", "attention_weights", "dense_masked_attention_bruteforce",
    "RopeConfig", "continuation_time_shift", "rope_inv_freq", "rope_angles", "rope_apply",
    "video_axis_split",
    "axis_window_count", "window_count", "window_ids", "window_partition", "window_pack",
    "window_unpack", "vsa_block_counts", "vsa_block_count", "vsa_block_ids", "vsa_block_means",
    "vsa_block_scores", "vsa_select", "vsa_attention", "ContinuationPlan", "continuation_plan",
    "continuation_pack", "continuation_append", "masked_update",
]
