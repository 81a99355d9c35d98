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
// Window attention straight on the (T, H, W) grid: windows of win[] cut with shift[] (edge
// windows cropped), frames_per_tile = 128 / (win[1] * win[2]) frames of a window per 128-row tile.
struct WindowAttnGeom {
  int L[3];
  int w[3];
  int s[3];
  int nwin[3];
  int frames_per_tile;
};

struct AttnArgs {
  // packed: 3-D views {D, H, capacity} of Q, K, V; window: 5-D views {D, H, W, Hgrid, T}
  CUtensorMap tmap_q, tmap_k, tmap_v;
  bool window;
  WindowAttnGeom wg;
  void* o;
  float* lse;
  const int32_t* cu_seqlens;
  int num_segments;
  int max_seqlen;
  int capacity;
  int num_heads;
  int head_dim;
  float scale;
  void* workspace;  // attn_workspace_bytes(num_segments) bytes: the work plan
  unsigned int* err;
};

size_t attn_workspace_bytes(int num_segments);
cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t stream);

}  // namespace h3
