// Shifted 3D window partition -> (perm, cu_seqlens) and the row gather / scatter around it.
//
// [H3-fast] "Breaking the engineering bottlenecks of video-generation models", "Breaking the
// memory wall: window attention across GPUs": the (T, H, W) token grid is cut into windows,
// alternate layers shift the window grid by half a window, edge windows are cropped to unequal
// sizes, and after attention the tokens are put back in their original order.
//
// The GPU enumerates directly: for a token (t, h, w) its axis windows are floor((x + s) / w);
// because window sizes factor per axis, the packed start of window (i_t, i_h, i_w) in
// lexicographic order is
//     P_t(i_t)*H*W + e_t(i_t)*P_h(i_h)*W + e_t(i_t)*e_h(i_h)*P_w(i_w)
// with P_a(i) = clamp(i*w_a - s_a, 0, L_a) the axis tokens before window i and
// e_a(i) = P_a(i+1) - P_a(i) its width; inside a window tokens keep row-major order.  No sort.
//
// The row copies are memory-bound: each row (H*D bf16) is read once and written once with
// 16-byte vectors, coalesced within the row.
#include "h3_internal.h"
#include "sm103_ptx.cuh"

namespace h3 {
namespace {

constexpr int kThreads = 256;
constexpr int kPackTokens = 16;  // rows per CTA
constexpr int kUnroll = 4;

__device__ __forceinline__ int axis_prefix(int i, int L, int w, int s) {
  const int v = i * w - s;
  return v < 0 ? 0 : (v > L ? L : v);
}

__device__ __forceinline__ int window_start(const WindowGeom& g, int it, int ih, int iw) {
  const int et = axis_prefix(it + 1, g.L[0], g.w[0], g.s[0]) - axis_prefix(it, g.L[0], g.w[0], g.s[0]);
  const int eh = axis_prefix(ih + 1, g.L[1], g.w[1], g.s[1]) - axis_prefix(ih, g.L[1], g.w[1], g.s[1]);
  return axis_prefix(it, g.L[0], g.w[0], g.s[0]) * g.L[1] * g.L[2] +
         et * axis_prefix(ih, g.L[1], g.w[1], g.s[1]) * g.L[2] +
         et * eh * axis_prefix(iw, g.L[2], g.w[2], g.s[2]);
}

__device__ __forceinline__ void copy_rows(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                          const int* s_src_row, const int* s_dst_row, int nrows,
                                          int row_vec) {
  const int total = nrows * row_vec;
#pragma unroll 1
  for (int v0 = threadIdx.x; v0 < total; v0 += kUnroll * kThreads) {
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kThreads;
      if (v < total) {
        const int i = v / row_vec;
        x[u] = __ldcs(src + static_cast<size_t>(s_src_row[i]) * row_vec + (v - i * row_vec));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * kThreads;
      if (v < total) {
        const int i = v / row_vec;
        if (s_dst_row[i] >= 0)
          __stcs(dst + static_cast<size_t>(s_dst_row[i]) * row_vec + (v - i * row_vec), x[u]);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads)
window_pack_kernel(const __grid_constant__ WindowGeom g, int32_t* __restrict__ perm,
                   int32_t* __restrict__ cu, const __grid_constant__ PackPtrs ptrs, int num_tensors, int row_vec, int num_tokens,
                   int num_windows) {
  __shared__ int s_src[kPackTokens];
  __shared__ int s_dst[kPackTokens];

  // cu_seqlens: window ids [blockIdx.x * kThreads, +kThreads)
  {
    const int id = blockIdx.x * kThreads + threadIdx.x;
    if (id < num_windows) {
      const int iw = id % g.nwin[2];
      const int ih = (id / g.nwin[2]) % g.nwin[1];
      const int it = id / (g.nwin[2] * g.nwin[1]);
      cu[id] = window_start(g, it, ih, iw);
    } else if (id == num_windows) {
      cu[id] = num_tokens;
    }
  }

  const int x0 = blockIdx.x * kPackTokens;
  if (x0 >= num_tokens) return;
  const int ntok = min(kPackTokens, num_tokens - x0);
  if (threadIdx.x < ntok) {
    const int x = x0 + threadIdx.x;
    const int HW = g.L[1] * g.L[2];
    const int t = x / HW;
    const int h = (x / g.L[2]) % g.L[1];
    const int w = x % g.L[2];
    const int it = (t + g.s[0]) / g.w[0];
    const int ih = (h + g.s[1]) / g.w[1];
    const int iw = (w + g.s[2]) / g.w[2];
    const int lo_t = axis_prefix(it, g.L[0], g.w[0], g.s[0]);
    const int lo_h = axis_prefix(ih, g.L[1], g.w[1], g.s[1]);
    const int lo_w = axis_prefix(iw, g.L[2], g.w[2], g.s[2]);
    const int eh = axis_prefix(ih + 1, g.L[1], g.w[1], g.s[1]) - lo_h;
    const int ew = axis_prefix(iw + 1, g.L[2], g.w[2], g.s[2]) - lo_w;
    const int p = window_start(g, it, ih, iw) + ((t - lo_t) * eh + (h - lo_h)) * ew + (w - lo_w);
    perm[p] = x;
    s_src[threadIdx.x] = x;
    s_dst[threadIdx.x] = p;
  }
  __syncthreads();
#pragma unroll 1
  for (int i = 0; i < num_tensors; ++i)
    copy_rows(static_cast<const uint4*>(ptrs.src[i]), static_cast<uint4*>(ptrs.dst[i]), s_src,
              s_dst, ntok, row_vec);
}

__global__ void __launch_bounds__(kThreads)
window_unpack_kernel(const int32_t* __restrict__ perm, int num_tokens, const uint4* __restrict__ src,
                     uint4* __restrict__ dst, int row_vec, unsigned int* err) {
  __shared__ int s_src[kPackTokens];
  __shared__ int s_dst[kPackTokens];
  const int j0 = blockIdx.x * kPackTokens;
  const int ntok = min(kPackTokens, num_tokens - j0);
  if (threadIdx.x < ntok) {
    const int j = j0 + threadIdx.x;
    int p = perm[j];
    if (p < 0 || p >= num_tokens) {  // not a permutation entry: skip the row, report it
      record_error(err, kErrBadPerm);
      p = -1;
    }
    s_src[threadIdx.x] = j;
    s_dst[threadIdx.x] = p;
  }
  __syncthreads();
  copy_rows(src, dst, s_src, s_dst, ntok, row_vec);
}

}  // namespace

cudaError_t launch_window_pack(const WindowGeom& g, int32_t* perm, int32_t* cu_seqlens,
                               const PackPtrs& ptrs, int num_tensors, int row_bytes,
                               cudaStream_t stream) {
  const int n = g.L[0] * g.L[1] * g.L[2];
  const int nwin = g.nwin[0] * g.nwin[1] * g.nwin[2];
  const int grid_tok = (n + kPackTokens - 1) / kPackTokens;
  const int grid_win = (nwin + 1 + kThreads - 1) / kThreads;
  const int grid = grid_tok > grid_win ? grid_tok : grid_win;
  window_pack_kernel<<<grid, kThreads, 0, stream>>>(g, perm, cu_seqlens, ptrs, num_tensors,
                                                    row_bytes / 16, n, nwin);
  return cudaGetLastError();
}

cudaError_t launch_window_unpack(const int32_t* perm, int num_tokens, const void* src, void* dst,
                                 int row_bytes, unsigned int* err, cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int grid = (num_tokens + kPackTokens - 1) / kPackTokens;
  window_unpack_kernel<<<grid, kThreads, 0, stream>>>(perm, num_tokens,
                                                      static_cast<const uint4*>(src),
                                                      static_cast<uint4*>(dst), row_bytes / 16, err);
  return cudaGetLastError();
}

}  // namespace h3
