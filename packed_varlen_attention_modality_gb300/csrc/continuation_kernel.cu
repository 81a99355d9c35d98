// Continuation window: packing of the five row groups, overlap discard / append, target-only
// row update.  All three are HBM-bound row copies (16-byte vectors, grid-stride, 4 vectors in
// flight per thread); the group boundaries and source offsets come from the host-side plan.
//
// [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section "Crossing
// the time boundary": the tail conditions (the last 7 latent video frames, the audio tail cut on
// the 40 Hz boundary) are taken straight from the previous window's latents; the DiT sequence is
// (1) text / reference, (2) audio tail, (3) video tail, (4) new audio noise, (5) new video noise;
// only (4) and (5) are updated by the denoising steps; afterwards the new samples that overlap the
// tails in time are dropped and the rest is appended to the clip.
#include <cstdint>

#include "h3_internal.h"
#include "h3attn.h"

namespace h3 {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;

// Each group is one contiguous range of rows in its source and in the packed sequence, so the
// copy is five range copies addressed in 16-byte vectors (no per-vector division by the row size).
struct PackSrc {
  const uint4* base[5];   // first source vector of each group
  int64_t dst_vec[6];     // exclusive prefix of the groups' vectors in the packed sequence
};

__global__ void __launch_bounds__(kCopyThreads)
continuation_pack_kernel(PackSrc src, ContinuationGeom g, uint4* __restrict__ out,
                         float* __restrict__ pos, uint8_t* __restrict__ tag,
                         uint8_t* __restrict__ target) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // positions, tags and the target mask, one thread per row (written first: the copy below
  // keeps every thread busy to the end)
  for (int64_t r64 = tid; r64 < g.num_rows; r64 += stride) {
    const int r = static_cast<int>(r64);
    int grp = 0;
#pragma unroll
    for (int k = 1; k < 5; ++k) grp += r >= g.offset[k];
    const int i = r - g.offset[grp];
    float t = static_cast<float>(i), h = 0.f, w = 0.f;
    uint8_t tg = H3_TAG_TEXT;
    if (grp == 1 || grp == 3) {
      tg = H3_TAG_AUDIO;
    } else if (grp == 2 || grp == 4) {  // (t, h, w) of a row-major frame grid
      const int hw = g.frame_h * g.frame_w;
      t = static_cast<float>(i / hw);
      h = static_cast<float>((i % hw) / g.frame_w);
      w = static_cast<float>(i % g.frame_w);
      tg = H3_TAG_VIDEO;
    }
    pos[3 * r64] = t;
    pos[3 * r64 + 1] = h;
    pos[3 * r64 + 2] = w;
    tag[r64] = tg;
    target[r64] = grp >= 3 ? 1 : 0;
  }
  const int64_t total = src.dst_vec[5];
  for (int64_t v0 = tid; v0 < total; v0 += stride * kUnroll) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < total) {
        int grp = 0;
#pragma unroll
        for (int k = 1; k < 5; ++k) grp += v >= src.dst_vec[k];
        buf[u] = __ldcs(src.base[grp] + (v - src.dst_vec[grp]));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < total) __stcs(out + v, buf[u]);
    }
  }
}

// Up to two contiguous row ranges copied in one launch (dst rows d0.., src rows s0..).
struct CopyRanges {
  const uint4* src[2];
  uint4* dst[2];
  int64_t vecs[2];  // 16-byte vectors of each range
};

__global__ void __launch_bounds__(kCopyThreads)
copy_ranges_kernel(CopyRanges c) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = c.vecs[0] + c.vecs[1];
  for (int64_t v0 = tid; v0 < total; v0 += stride * kUnroll) {
    uint4 buf[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < total) buf[u] = v < c.vecs[0] ? __ldcs(c.src[0] + v) : __ldcs(c.src[1] + (v - c.vecs[0]));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < total) {
        if (v < c.vecs[0]) __stcs(c.dst[0] + v, buf[u]);
        else __stcs(c.dst[1] + (v - c.vecs[0]), buf[u]);
      }
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads)
masked_row_update_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                         const uint8_t* __restrict__ mask, int num_rows, int vec_per_row) {
  const int64_t total = static_cast<int64_t>(num_rows) * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t v = tid; v < total; v += stride) {
    if (__ldg(mask + v / vec_per_row)) __stcs(dst + v, __ldcs(src + v));
  }
}

int copy_grid(int64_t vecs) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  const int64_t want = (vecs + kCopyThreads * kUnroll - 1) / (kCopyThreads * kUnroll);
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 CTAs of 256 threads per SM
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_continuation_pack(const ContinuationGeom& g, const void* const src[5],
                                     const int64_t first_row[5], int row_bytes, void* rows,
                                     float* pos, uint8_t* tag, uint8_t* target,
                                     cudaStream_t stream) {
  if (g.num_rows <= 0) return cudaSuccess;
  const int64_t vpr = row_bytes / 16;
  PackSrc s;
  for (int k = 0; k < 5; ++k) {
    s.base[k] = src[k] == nullptr ? nullptr : static_cast<const uint4*>(src[k]) + first_row[k] * vpr;
    s.dst_vec[k] = static_cast<int64_t>(g.offset[k]) * vpr;
  }
  s.dst_vec[5] = static_cast<int64_t>(g.num_rows) * vpr;
  continuation_pack_kernel<<<copy_grid(s.dst_vec[5]), kCopyThreads, 0, stream>>>(
      s, g, static_cast<uint4*>(rows), pos, tag, target);
  return cudaGetLastError();
}

cudaError_t launch_copy_ranges(const void* const src[2], void* const dst[2], const int64_t bytes[2],
                               cudaStream_t stream) {
  CopyRanges c;
  for (int k = 0; k < 2; ++k) {
    c.src[k] = static_cast<const uint4*>(src[k]);
    c.dst[k] = static_cast<uint4*>(dst[k]);
    c.vecs[k] = bytes[k] / 16;
  }
  if (c.vecs[0] + c.vecs[1] == 0) return cudaSuccess;
  copy_ranges_kernel<<<copy_grid(c.vecs[0] + c.vecs[1]), kCopyThreads, 0, stream>>>(c);
  return cudaGetLastError();
}

cudaError_t launch_masked_row_update(void* dst, const void* src, const uint8_t* mask, int num_rows,
                                     int row_bytes, cudaStream_t stream) {
  if (num_rows <= 0) return cudaSuccess;
  const int vpr = row_bytes / 16;
  masked_row_update_kernel<<<copy_grid(static_cast<int64_t>(num_rows) * vpr), kCopyThreads, 0,
                             stream>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                       mask, num_rows, vpr);
  return cudaGetLastError();
}

}  // namespace h3
