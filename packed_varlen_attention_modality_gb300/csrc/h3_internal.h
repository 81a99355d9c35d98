// Host-side launchers shared between the C-ABI translation unit and the kernel translation units.
// Arguments arrive already validated by h3attn_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace h3 {

// ---- RoPE ---------------------------------------------------------------------------------
constexpr int kMaxPairs = 64;  // head_dim <= 128

// Per-pair fp32 inverse frequencies (computed on the host in fp64, rounded once) and, for video
// rows, which coordinate drives each pair (0 = t, 1 = h, 2 = w).
struct RopeTables {
  float inv_text[kMaxPairs];
  float inv_audio[kMaxPairs];
  float inv_video[kMaxPairs];
  uint8_t video_axis[kMaxPairs];
  float audio_hz;
  float video_fps;
};

cudaError_t launch_rope(const void* q_in, void* q_out, const void* k_in, void* k_out,
                        int num_tokens, int num_heads, int head_dim, const float* pos,
                        const uint8_t* tag, const int32_t* cu_requests, int num_requests,
                        const float* start_frames, const RopeTables& tables, cudaStream_t stream);

// ---- window partition ---------------------------------------------------------------------
struct WindowGeom {
  int L[3];      // grid extent per axis (T, H, W)
  int w[3];      // window size per axis
  int s[3];      // shift per axis
  int nwin[3];   // axis window counts
};

constexpr int kMaxPackTensors = 8;
struct PackPtrs {
  const void* src[kMaxPackTensors];
  void* dst[kMaxPackTensors];
};

cudaError_t launch_window_pack(const WindowGeom& g, int32_t* perm, int32_t* cu_seqlens,
                               const PackPtrs& ptrs, int num_tensors, int row_bytes,
                               cudaStream_t stream);
cudaError_t launch_window_unpack(const int32_t* perm, int num_tokens, const void* src, void* dst,
                                 int row_bytes, unsigned int* err, cudaStream_t stream);

// ---- attention ------------------------------------------------------------------------------
// Attention kernel variants: packed varlen segments; 3D windows read in place on the grid;
// block-sparse video attention over selected 64-token blocks read in place on the grid.
constexpr int kAttnModePacked = 0;
constexpr int kAttnModeWindow = 1;
constexpr int kAttnModeVsa = 2;

// Attention straight on the (T, H, W) grid.
// Windows: windows of w[] cut with shift s[] (edge windows cropped), nwin[] windows per axis,
// frames_per_tile = 128 / (w[1] * w[2]) frames of a window per 128-row tile.
// VSA: blocks of w[] (w[0] * w[1] * w[2] = 64) cut without shift (s = 0), nwin[] blocks per axis,
// topk selected key blocks per query block.
struct WindowAttnGeom {
  int L[3];
  int w[3];
  int s[3];
  int nwin[3];
  int frames_per_tile;
  int half_h;  // windows: half-height maps exist (window H even) for edge windows
  int topk;
};

struct AttnArgs {
  // packed: 3-D views {D, H, capacity} of Q, K, V; window: 5-D views {D, H, W, Hgrid, T}
  CUtensorMap tmap_q, tmap_k, tmap_v;
  // window: the same views with half-height boxes (edge windows); otherwise copies of the above
  CUtensorMap tmap_q2, tmap_k2, tmap_v2;
  int mode;            // kAttnModePacked / kAttnModeWindow / kAttnModeVsa
  WindowAttnGeom wg;
  // VSA: the key/value steps of every (head, pair of query blocks), from launch_vsa_schedule
  const uint2* vsa_steps;
  const int2* vsa_counts;
  void* o;
  float* lse;
  const int32_t* cu_seqlens;
  int num_segments;
  int max_seqlen;
  int capacity;
  int num_heads;
  int head_dim;
  float scale;
  void* workspace;  // attn_plan_bytes(num_segments) bytes: the work plan
  void* split_area;  // packed: attn_split_bytes(head_dim) bytes after the plan, or null (no split)
  unsigned int* err;
  uint64_t wait_limit_ns;  // limit of the kernel's pipeline waits (wait_limit_ns() below)
  uint32_t stall_after_tiles;  // testing hook: producers stop after this many K/V tiles
};

// Limit of the attention kernels' pipeline waits for launches from now on: 2 s unless
// h3_set_wait_limit_ns changed it.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
uint64_t wait_limit_ns();
// Key/value tiles a producer of an attention CTA issues before it stops (all, unless
// h3_debug_stall_loads changed it).
uint32_t stall_after_tiles();

// Workspace of the packed variant.  The plan (uint32 words): [0] split items, [1] work items, [2] whole items
// before the split last wave, [3] entries of that wave, [kAttnWsHeaderWords, +S) segment order,
// [kAttnWsHeaderWords + S, +S+1) exclusive prefix of whole items in that order; rounded up to
// 256 bytes.  Then, optionally, the split area of the last wave (entries, arrival counters and
// partial results of up to kSplitMaxEntries chunks): with it the call may cut the long items of
// its last wave into chunks of their key range; without it every item stays whole.
constexpr int kAttnWsHeaderWords = 4;
constexpr int kSplitMaxEntries = 320;  // chunks of the last wave (>= 2 x 152 SMs)
constexpr int kSplitMinSeqlen = 1024;  // the area is only asked for when a segment can be this long
constexpr size_t attn_plan_bytes(int num_segments) {
  return ((kAttnWsHeaderWords + 2 * static_cast<size_t>(num_segments) + 1) * sizeof(uint32_t) + 255) /
         256 * 256;
}
// entries (8 words each), a list of split items (one word each), then per entry and query tile
// 128 rows of head_dim fp32 values followed by their 128 fp32 LSEs
constexpr size_t attn_split_bytes(int head_dim) {
  return static_cast<size_t>(kSplitMaxEntries) * (8 + 1) * sizeof(uint32_t) +
         static_cast<size_t>(kSplitMaxEntries) * 2 * 128 * (head_dim + 1) * sizeof(float);
}
constexpr size_t attn_workspace_bytes(int num_segments, int max_seqlen, int head_dim) {
  return attn_plan_bytes(num_segments) + (max_seqlen >= kSplitMinSeqlen ? attn_split_bytes(head_dim) : 0);
}
cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t stream);

// ---- VSA block gate + top-k ----------------------------------------------------------------
struct VsaGeom {
  int L[3];   // grid (T, H, W)
  int b[3];   // block size per axis
  int nb[3];  // blocks per axis = ceil(L / b)
};
// Workspace: block means of Q and K, fp32 [2][heads][nblk][head_dim].
size_t vsa_pool_bytes(int nblk, int heads, int head_dim);
// scores: fp32 [heads, nblk, nblk] out; sel: int32 [heads, nblk, topk] out (ascending ids).
cudaError_t launch_vsa_select(const void* q, const void* k, const VsaGeom& g, int heads,
                              int head_dim, int topk, float scale, float* scores, int32_t* sel,
                              void* workspace, cudaStream_t stream);

// VSA key/value schedule.  Query blocks 2p and 2p + 1 (the two halves of one 128-row tile; the
// second is block 2p again past the last block) form pair p.  Step j of pair p loads two key
// blocks into the two 64-row halves of a key tile: steps[(h * npairs + p) * topk + j] holds
// {block of half 0 | use0 << kVsaUseShift, block of half 1 | use1 << kVsaUseShift}, where bit q
// of use_s says whether query block 2p + q attends to that half's keys.  counts[h * npairs + p]
// = {steps used (<= topk), s = blocks both query blocks selected}.  The steps follow a fixed
// layout: s / 2 steps of two shared blocks (both halves used by both), one step with the odd
// shared block in half 0 when s is odd, then steps whose half q is query block 2p + q's own.
constexpr int kVsaUseShift = 28;
constexpr uint32_t kVsaBlockMask = (1u << kVsaUseShift) - 1u;
inline int vsa_pairs(int nblk) { return (nblk + 1) / 2; }
size_t vsa_schedule_bytes(int nblk, int heads, int topk);
// sel: int32 [heads, nblk, topk]; workspace: vsa_schedule_bytes() bytes, 16-byte aligned.
cudaError_t launch_vsa_schedule(const int32_t* sel, int nblk, int heads, int topk, void* workspace,
                                unsigned int* err, cudaStream_t stream);

// ---- continuation window ---------------------------------------------------------------------
struct ContinuationGeom {
  int offset[5];  // first packed row of each group (offset[0] = 0)
  int num_rows;
  int frame_h, frame_w;  // latent grid of a video frame
};
// src[k]: device base of group k's source rows; first_row[k]: its first source row.
cudaError_t launch_continuation_pack(const ContinuationGeom& g, const void* const src[5],
                                     const int64_t first_row[5], int row_bytes, void* rows,
                                     float* pos, uint8_t* tag, uint8_t* target, cudaStream_t stream);
// Two contiguous device copies (bytes multiples of 16, 16-byte aligned) in one launch.
cudaError_t launch_copy_ranges(const void* const src[2], void* const dst[2], const int64_t bytes[2],
                               cudaStream_t stream);
cudaError_t launch_masked_row_update(void* dst, const void* src, const uint8_t* mask, int num_rows,
                                     int row_bytes, cudaStream_t stream);

}  // namespace h3
