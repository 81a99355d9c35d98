// Block-sparse video attention (VSA): block gate scores and top-k block selection on sm_103a.
//
// [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section "VSA:
// block-sparse attention": the video latent is cut into 4x4x4 = 64-token blocks along time,
// height and width; a block-level gate scores every key block against the current query block
// and only the top-k blocks take part in the token-level attention (the attention itself is the
// kModeVsa variant of attn_fwd_sm103.cu).  The gate here is the scaled dot product of the block
// means (no learned gate is given); equal scores prefer the lower block id; the selected ids are
// written in ascending order.
//
// Three kernels, all HBM- or FFMA-bound (the gate is ~1 % of the fine attention's work):
//   vsa_pool_kernel    mean of each block's Q and K rows per head (fp32 sums in token order)
//   vsa_score_kernel   S_h = scale * Qmean_h Kmean_h^T, a 64 x 128 output tile per CTA with
//                      8 x 4 register micro-tiles (two broadcast and one float4 shared loads per
//                      32 FFMA), written to the caller's [H, nblk, nblk] score buffer
//   vsa_topk_kernel    one warp per (head, query block): 8-bit radix select of the k-th largest
//                      score over 4 passes (the row stays in L1/L2), then an ascending ballot
//                      compaction that takes the ties at the threshold lowest id first
//
// And the attention's key/value schedule (vsa_schedule_kernel, one warp per head and pair of
// query blocks).  The token-level attention runs a 128-row query tile as two query blocks, one
// per 64-row half, and each step loads a 128-row key tile as two key blocks.  A block that both
// query blocks selected serves both halves, so two such blocks fill a step with no masked work;
// a block only one of them selected is paired with one only the other selected, as before.  With
// s shared selections a pair takes ceil(s / 2) + (topk - s) steps instead of topk.  Sorted lists
// (as vsa_topk_kernel writes them) are intersected as multisets by binary search; lists in any
// other order, or with an id out of range (recorded, then read as block 0), keep one step per
// list entry.
#include <cuda_bf16.h>

#include <atomic>

#include <cstdint>

#include "h3_internal.h"
#include "sm103_ptx.cuh"

namespace h3 {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kScoreRows = 64;     // query blocks per score tile
constexpr int kScoreCols = 128;    // key blocks per score tile
constexpr int kScoreThreads = 256;
constexpr int kTopkWarps = 8;
constexpr int kSchedWarps = 8;

// Block b of the grid: origin and extent (cropped by the grid edge).
struct BlockBox {
  int t0, h0, w0, nt, nh, nw;
};
__device__ __forceinline__ BlockBox block_box(int b, const VsaGeom& g) {
  BlockBox x;
  const int iw = b % g.nb[2], ih = (b / g.nb[2]) % g.nb[1], it = b / (g.nb[2] * g.nb[1]);
  x.t0 = it * g.b[0];
  x.h0 = ih * g.b[1];
  x.w0 = iw * g.b[2];
  x.nt = min(g.b[0], g.L[0] - x.t0);
  x.nh = min(g.b[1], g.L[1] - x.h0);
  x.nw = min(g.b[2], g.L[2] - x.w0);
  return x;
}

// grid (nblk, 2): blockIdx.y selects Q (0) or K (1).  Each thread owns 8 consecutive elements of
// the H*D token row and sums the block's rows in row-major token order.
__global__ void __launch_bounds__(kPoolThreads)
vsa_pool_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                VsaGeom g, int heads, int head_dim, float* __restrict__ qm,
                float* __restrict__ km) {
  const int b = blockIdx.x;
  const __nv_bfloat16* src = blockIdx.y == 0 ? q : k;
  float* dst = blockIdx.y == 0 ? qm : km;
  const BlockBox x = block_box(b, g);
  const int row_elems = heads * head_dim;
  const float inv = 1.f / static_cast<float>(x.nt * x.nh * x.nw);
  const int nblk = g.nb[0] * g.nb[1] * g.nb[2];
  for (int e0 = threadIdx.x * 8; e0 < row_elems; e0 += kPoolThreads * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int ft = 0; ft < x.nt; ++ft)
      for (int fh = 0; fh < x.nh; ++fh)
        for (int fw = 0; fw < x.nw; ++fw) {
          const size_t tok =
              (static_cast<size_t>(x.t0 + ft) * g.L[1] + (x.h0 + fh)) * g.L[2] + (x.w0 + fw);
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + tok * row_elems + e0));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
          }
        }
    // element e = h * D + d  ->  dst[h][b][d]
    const int h = e0 / head_dim, d = e0 % head_dim;
    float4* o = reinterpret_cast<float4*>(dst + (static_cast<size_t>(h) * nblk + b) * head_dim + d);
    o[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    o[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
}

// grid (ceil(nblk / 128), ceil(nblk / 64), heads).  Thread (rg, kg) = (tid / 32, tid % 32)
// computes query blocks 8 rg .. 8 rg + 7 against key blocks 4 kg .. 4 kg + 3 of the tile: per
// dimension two broadcast and one conflict-free float4 shared load feed 32 FFMA.  The tile's
// operands (102 KB at D = 128) leave room for two CTAs per SM, so one CTA's loads overlap the
// other's FFMA (a 64 x 256 tile, one CTA per SM, kept the FMA pipes 27 % busy).
constexpr int kQs = kScoreRows + 4;  // padded smem row lengths (float4 alignment kept)
constexpr int kKs = kScoreCols + 4;
template <int D>
constexpr int score_smem_bytes() {
  return D * (kQs + kKs) * static_cast<int>(sizeof(float));
}

template <int D>
__global__ void __launch_bounds__(kScoreThreads)
vsa_score_kernel(const float* __restrict__ qm, const float* __restrict__ km, int nblk, float scale,
                 float* __restrict__ scores) {
  extern __shared__ __align__(16) float score_smem[];
  float* qs = score_smem;           // [d][row]
  float* ks = score_smem + D * kQs;  // [d][col]
  const int h = blockIdx.z;
  const int r0 = blockIdx.y * kScoreRows, c0 = blockIdx.x * kScoreCols;
  const float* qh = qm + static_cast<size_t>(h) * nblk * D;
  const float* kh = km + static_cast<size_t>(h) * nblk * D;
  for (int i = threadIdx.x; i < kScoreRows * D; i += kScoreThreads) {
    const int r = i / D, d = i % D;
    qs[d * kQs + r] = r0 + r < nblk ? qh[static_cast<size_t>(r0 + r) * D + d] : 0.f;
  }
  for (int i = threadIdx.x; i < kScoreCols * D; i += kScoreThreads) {
    const int c = i / D, d = i % D;
    ks[d * kKs + c] = c0 + c < nblk ? kh[static_cast<size_t>(c0 + c) * D + d] : 0.f;
  }
  __syncthreads();
  const int rg = threadIdx.x >> 5, kg = threadIdx.x & 31;
  float acc[8][4] = {};
#pragma unroll 4
  for (int d = 0; d < D; ++d) {
    const float4 a0 = *reinterpret_cast<const float4*>(&qs[d * kQs + 8 * rg]);
    const float4 a1 = *reinterpret_cast<const float4*>(&qs[d * kQs + 8 * rg + 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&ks[d * kKs + 4 * kg]);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[4] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + 8 * rg + i;
    if (r >= nblk) break;
    float* row = scores + (static_cast<size_t>(h) * nblk + r) * nblk;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + 4 * kg + j;
      if (c < nblk) row[c] = acc[i][j] * scale;
    }
  }
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per (head, query block) row of the score matrix.  The five passes re-read the row
// (8 KB at 2016 blocks) through L1/L2: with only the 8 KB histogram in shared memory, enough
// warps stay resident to hide the latency (staging rows in shared memory was slower).
__global__ void __launch_bounds__(kTopkWarps * 32)
vsa_topk_kernel(const float* __restrict__ scores, int rows, int nblk, int topk,
                int32_t* __restrict__ sel) {
  __shared__ uint32_t hist_all[kTopkWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kTopkWarps + warp;
  if (row >= rows) return;
  uint32_t* hist = hist_all[warp];
  const float* s = scores + static_cast<size_t>(row) * nblk;
  // radix select of the topk-th largest key, 8 bits per pass from the top
  uint32_t prefix = 0, mask = 0;
  int remaining = topk;  // how many of the wanted keys still lie at or below the current prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0u;
    __syncwarp();
    for (int i = lane; i < nblk; i += 32) {
      const uint32_t key = order_key(s[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane L holds bins 255 - 8L down to 248 - 8L; find the bin where the count from the top
    // reaches `remaining`
    uint32_t mine[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mine[i] = hist[255 - 8 * lane - i];
      sum += mine[i];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const uint32_t excl = incl - sum;
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= static_cast<uint32_t>(remaining));
    const int src = __ffs(hit) - 1;  // the first lane whose running count reaches it
    int bin = 0, above = 0;
    if (lane == src) {
      uint32_t run = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (run + mine[i] >= static_cast<uint32_t>(remaining)) {
          bin = 255 - 8 * lane - i;
          above = static_cast<int>(run);
          break;
        }
        run += mine[i];
      }
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    above = __shfl_sync(0xffffffffu, above, src);
    remaining -= above;
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  // prefix is the threshold key; `remaining` of the keys equal to it are taken, lowest id first
  int32_t* out = sel + static_cast<size_t>(row) * topk;
  int taken = 0, eq_seen = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = 0; i0 < nblk; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < nblk ? order_key(s[i]) : 0u;
    const bool gt = i < nblk && key > prefix;
    const bool eq = i < nblk && key == prefix;
    const unsigned eq_mask = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_seen + __popc(eq_mask & lt) < remaining);
    const unsigned take_mask = __ballot_sync(0xffffffffu, take);
    if (take) out[taken + __popc(take_mask & lt)] = i;
    taken += __popc(take_mask);
    eq_seen += __popc(eq_mask);
  }
}

// First index in a[0, n) whose value is >= x (a ascending).
__device__ __forceinline__ int lower_idx(const int32_t* __restrict__ a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}
// Entries equal to x in a[0, n) (a ascending).
__device__ __forceinline__ int count_of(const int32_t* __restrict__ a, int n, int x) {
  const int lo = lower_idx(a, n, x);
  int hi = n, l = lo;
  while (l < hi) {
    const int mid = (l + hi) >> 1;
    if (__ldg(a + mid) <= x) l = mid + 1; else hi = mid;
  }
  return l - lo;
}

__global__ void __launch_bounds__(kSchedWarps * 32)
vsa_schedule_kernel(const int32_t* __restrict__ sel, int nblk, int heads, int topk,
                    uint32_t* __restrict__ steps, int2* __restrict__ counts, unsigned int* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npairs = (nblk + 1) / 2;
  const int pid = blockIdx.x * kSchedWarps + warp;  // h * npairs + p
  if (pid >= heads * npairs) return;
  const int h = pid / npairs, p = pid % npairs;
  const int32_t* A = sel + (static_cast<size_t>(h) * nblk + 2 * p) * topk;
  const int32_t* B = sel + (static_cast<size_t>(h) * nblk + min(2 * p + 1, nblk - 1)) * topk;
  uint32_t* out = steps + static_cast<size_t>(pid) * topk * 2;  // [topk][half]
  const unsigned lt = (1u << lane) - 1u;
  bool valid = true, sorted = true;
  for (int i = lane; i < topk; i += 32) {
    const int a = __ldg(A + i), b = __ldg(B + i);
    valid = valid && a >= 0 && a < nblk && b >= 0 && b < nblk;
    if (i > 0) sorted = sorted && __ldg(A + i - 1) <= a && __ldg(B + i - 1) <= b;
  }
  valid = __all_sync(0xffffffffu, valid);
  sorted = __all_sync(0xffffffffu, sorted);
  if (!valid && lane == 0) record_error(err, kErrBadBlockIndex);
  if (!valid || !sorted) {
    for (int j = lane; j < topk; j += 32) {
      int a = __ldg(A + j), b = __ldg(B + j);
      if (a < 0 || a >= nblk) a = 0;
      if (b < 0 || b >= nblk) b = 0;
      out[2 * j] = static_cast<uint32_t>(a) | (1u << kVsaUseShift);
      out[2 * j + 1] = static_cast<uint32_t>(b) | (2u << kVsaUseShift);
    }
    if (lane == 0) counts[pid] = make_int2(topk, 0);
    return;
  }
  // entry i of A is shared when fewer copies of its id precede it in A than B holds (and the
  // other way round for B): the multiset intersection, taken in list order
  auto shared_a = [&](int i) {
    const int x = __ldg(A + i);
    return i - lower_idx(A, i, x) < count_of(B, topk, x);
  };
  auto shared_b = [&](int j) {
    const int y = __ldg(B + j);
    return j - lower_idx(B, j, y) < count_of(A, topk, y);
  };
  int ns = 0;
  for (int i0 = 0; i0 < topk; i0 += 32) {
    const int i = i0 + lane;
    ns += __popc(__ballot_sync(0xffffffffu, i < topk && shared_a(i)));
  }
  const int s0 = (ns + 1) / 2;  // steps of shared blocks
  // shared blocks two per step, both halves; then A's own blocks in half 0 beside B's own in half 1
  int nc = 0, na = 0;
  for (int i0 = 0; i0 < topk; i0 += 32) {
    const int i = i0 + lane;
    const bool in = i < topk;
    const bool c = in && shared_a(i);
    const unsigned cm = __ballot_sync(0xffffffffu, c), am = __ballot_sync(0xffffffffu, in && !c);
    if (in) {
      const uint32_t x = static_cast<uint32_t>(__ldg(A + i));
      if (c) {
        const int r = nc + __popc(cm & lt);
        out[2 * (r >> 1) + (r & 1)] = x | (3u << kVsaUseShift);
        if (r == ns - 1 && (ns & 1)) out[2 * (r >> 1) + 1] = x;  // odd one out: other half unused
      } else {
        out[2 * (s0 + na + __popc(am & lt))] = x | (1u << kVsaUseShift);
      }
    }
    nc += __popc(cm);
    na += __popc(am);
  }
  int nb = 0;
  for (int j0 = 0; j0 < topk; j0 += 32) {
    const int j = j0 + lane;
    const bool own = j < topk && !shared_b(j);
    const unsigned bm = __ballot_sync(0xffffffffu, own);
    if (own)
      out[2 * (s0 + nb + __popc(bm & lt)) + 1] = static_cast<uint32_t>(__ldg(B + j)) | (2u << kVsaUseShift);
    nb += __popc(bm);
  }
  if (lane == 0) counts[pid] = make_int2(s0 + (topk - ns), ns);
}

template <int D>
cudaError_t launch_score(dim3 grid, const float* qm, const float* km, int nblk, float scale,
                         float* scores, cudaStream_t stream) {
  // the shared-memory opt-in is made once per device (a second call from a racing thread is
  // harmless; the flags are atomic so the race is defined)
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(vsa_score_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             score_smem_bytes<D>());
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  vsa_score_kernel<D><<<grid, kScoreThreads, score_smem_bytes<D>(), stream>>>(qm, km, nblk, scale,
                                                                              scores);
  return cudaGetLastError();
}

}  // namespace

size_t vsa_schedule_bytes(int nblk, int heads, int topk) {
  const size_t pairs = static_cast<size_t>(heads) * vsa_pairs(nblk);
  return (pairs * topk * 8 + 255) / 256 * 256 + (pairs * 8 + 255) / 256 * 256;
}

cudaError_t launch_vsa_schedule(const int32_t* sel, int nblk, int heads, int topk, void* workspace,
                                unsigned int* err, cudaStream_t stream) {
  const size_t pairs = static_cast<size_t>(heads) * vsa_pairs(nblk);
  uint32_t* steps = static_cast<uint32_t*>(workspace);
  int2* counts = reinterpret_cast<int2*>(static_cast<uint8_t*>(workspace) +
                                         (pairs * topk * 8 + 255) / 256 * 256);
  const unsigned blocks = static_cast<unsigned>((pairs + kSchedWarps - 1) / kSchedWarps);
  vsa_schedule_kernel<<<blocks, kSchedWarps * 32, 0, stream>>>(sel, nblk, heads, topk, steps,
                                                               counts, err);
  return cudaGetLastError();
}

size_t vsa_pool_bytes(int nblk, int heads, int head_dim) {
  const size_t b = 2ull * heads * nblk * head_dim * sizeof(float);
  return (b + 255) / 256 * 256;
}

cudaError_t launch_vsa_select(const void* q, const void* k, const VsaGeom& g, int heads,
                              int head_dim, int topk, float scale, float* scores, int32_t* sel,
                              void* workspace, cudaStream_t stream) {
  const int nblk = g.nb[0] * g.nb[1] * g.nb[2];
  float* qm = static_cast<float*>(workspace);
  float* km = qm + static_cast<size_t>(heads) * nblk * head_dim;
  vsa_pool_kernel<<<dim3(nblk, 2), kPoolThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g, heads,
      head_dim, qm, km);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 sgrid((nblk + kScoreCols - 1) / kScoreCols, (nblk + kScoreRows - 1) / kScoreRows,
                   heads);
  e = head_dim == 128 ? launch_score<128>(sgrid, qm, km, nblk, scale, scores, stream)
                      : launch_score<64>(sgrid, qm, km, nblk, scale, scores, stream);
  if (e != cudaSuccess) return e;
  const int rows = heads * nblk;
  vsa_topk_kernel<<<(rows + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, stream>>>(
      scores, rows, nblk, topk, sel);
  return cudaGetLastError();
}

}  // namespace h3
