// Modality-tagged rotary position encoding with the continuation time shift.
//
// [H3-vLLM] "Joint audio/video generation in production: MiniMax-H3 and vLLM-Omni", sec. 3:
// each token's modality tag selects its RoPE frequencies; modality position spaces are
// independent.  [H3-fast] "Crossing the time boundary", step 3: t_global = t_local + s*40/24 is
// applied to the time coordinate only, before the encoding.
//
// Memory-bound: every Q/K element is read once and written once.  A CTA owns kTokens
// consecutive tokens; it first computes the (cos, sin) of each (token, pair) once into shared
// memory (shared by all heads and by Q and K), then streams the tokens' Q and K rows through in
// 16-byte vectors (8 bf16 = 4 rotation pairs), fully coalesced.
#include <cuda_bf16.h>

#include "h3_internal.h"
#include "sm103_ptx.cuh"

namespace h3 {
namespace {

constexpr int kThreads = 256;
constexpr int kTokens = 4;
constexpr int kUnroll = 4;

__device__ __forceinline__ int request_of(const int32_t* __restrict__ cu_requests, int num_requests,
                                          int n) {
  // largest r in [0, num_requests) with cu_requests[r] <= n
  int lo = 0, hi = num_requests - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_requests[mid] <= n) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint4 rotate4(uint4 x, const float2* __restrict__ cs) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w[p]);
    const float2 f = __bfloat1622float2(b);
    const float2 r = cs[p];  // (cos, sin)
    const float y0 = fmaf(f.x, r.x, -f.y * r.y);
    const float y1 = fmaf(f.x, r.y, f.y * r.x);
    b = __floats2bfloat162_rn(y0, y1);
    w[p] = *reinterpret_cast<uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kThreads)
rope_kernel(const uint4* q_in, uint4* q_out, const uint4* k_in, uint4* k_out,
            int num_tokens, int num_heads, int head_dim, const float* __restrict__ pos,
            const uint8_t* __restrict__ tag, const int32_t* __restrict__ cu_requests,
            int num_requests, const float* __restrict__ start_frames,
            const __grid_constant__ RopeTables tab) {
  __shared__ float2 cs[kTokens][kMaxPairs];
  // Nothing of what this kernel writes (Q and K) is read by the plan kernel that may follow it:
  // let that kernel be scheduled now (it waits for this grid before reading anything).
  launch_dependents();
  const int tok0 = blockIdx.x * kTokens;
  const int ntok = min(kTokens, num_tokens - tok0);
  const int P = head_dim >> 1;

  // (1) angles: one (token, pair) per thread, shared by all heads and by Q and K
  for (int idx = threadIdx.x; idx < ntok * P; idx += kThreads) {
    const int ti = idx / P;
    const int j = idx - ti * P;
    const int n = tok0 + ti;
    const int tg = tag[n];
    float t = pos[3 * n];
    if (start_frames != nullptr) {
      const int r = (cu_requests != nullptr) ? request_of(cu_requests, num_requests, n) : 0;
      // s * 40 / 24 with one correctly rounded division (s*40 is exact for integral s < 2^18)
      t = t + __fdiv_rn(start_frames[r] * tab.audio_hz, tab.video_fps);
    }
    float coord, inv;
    if (tg == 1) {  // video: the pair's band picks t, h or w
      const int axis = tab.video_axis[j];
      coord = (axis == 0) ? t : pos[3 * n + axis];
      inv = tab.inv_video[j];
    } else if (tg == 2) {  // audio
      coord = t;
      inv = tab.inv_audio[j];
    } else {  // text
      coord = t;
      inv = tab.inv_text[j];
    }
    float s, c;
    sincosf(coord * inv, &s, &c);
    cs[ti][j] = make_float2(c, s);
  }
  __syncthreads();

  // (2) rotate the CTA's rows of Q, then K
  const int vec_per_head = head_dim >> 3;
  const int vec_per_tok = num_heads * vec_per_head;
  const int total = ntok * vec_per_tok;
  const size_t base = static_cast<size_t>(tok0) * vec_per_tok;
#pragma unroll 1
  for (int tensor = 0; tensor < 2; ++tensor) {
    const uint4* src = tensor ? k_in : q_in;
    uint4* dst = tensor ? k_out : q_out;
    if (src == nullptr) break;
#pragma unroll 1
    for (int v0 = threadIdx.x; v0 < total; v0 += kUnroll * kThreads) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kThreads;
        if (v < total) x[u] = __ldcs(src + base + v);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kThreads;
        if (v < total) {
          const int ti = v / vec_per_tok;
          const int pr = (v % vec_per_head) * 4;
          __stcs(dst + base + v, rotate4(x[u], &cs[ti][pr]));
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope(const void* q_in, void* q_out, const void* k_in, void* k_out,
                        int num_tokens, int num_heads, int head_dim, const float* pos,
                        const uint8_t* tag, const int32_t* cu_requests, int num_requests,
                        const float* start_frames, const RopeTables& tables,
                        cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int grid = (num_tokens + kTokens - 1) / kTokens;
  rope_kernel<<<grid, kThreads, 0, stream>>>(
      static_cast<const uint4*>(q_in), static_cast<uint4*>(q_out),
      static_cast<const uint4*>(k_in), static_cast<uint4*>(k_out), num_tokens, num_heads,
      head_dim, pos, tag, cu_requests, num_requests, start_frames, tables);
  return cudaGetLastError();
}

}  // namespace h3
