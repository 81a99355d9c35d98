// C ABI of libh3attn: argument validation, tensor-map construction, kernel launch.
//
// Nothing here allocates device memory.  The one piece of library-owned device state is the
// error word below (a static __device__ variable, 4 bytes per device), where kernels record the
// first device-side problem they meet (bad cu_seqlens, bad permutation entry, a timed-out wait).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "h3attn.h"
#include "h3_internal.h"

// Scratch for h3_varlen_attn_fwd_noalloc: the attention work plan lives in this fixed array
// instead of a caller-provided workspace.  Every device that loads the library holds it (132 KB,
// enough for H3_NOALLOC_MAX_SEGMENTS segments) until the process exits.  It is shared by all
// calls on a device.
constexpr int kNoallocScratchBytes = 132 * 1024;
static_assert(h3::attn_plan_bytes(H3_NOALLOC_MAX_SEGMENTS) <= kNoallocScratchBytes,
              "the no-alloc array must hold the plan of H3_NOALLOC_MAX_SEGMENTS segments");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

namespace {

__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int* g_err_ptr[kMaxDevices] = {};

// Device address of g_device_error on the current device (looked up once per device).
unsigned int* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D view {D, H, rows} of a bf16 [rows, H, D] tensor; box {64, 1, 128}, 128-byte swizzle.
bool make_qkv_map(CUtensorMap* m, const void* base, int rows, int heads, int head_dim) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(heads) * head_dim * 2};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D view {D, heads, W, H, T} of a bf16 [T*H*W, heads, D] tensor in row-major token order; box
// {64, 1, win_w, win_h, frames} (one 128-row tile of a window), 128-byte swizzle.  Coordinates
// outside the grid (edge windows) read as zero.
bool make_window_map(CUtensorMap* m, const void* base, const int32_t grid[3], const int32_t win[3],
                     int frames, int heads, int head_dim) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(heads) * head_dim * 2;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(grid[2]), static_cast<cuuint64_t>(grid[1]),
                              static_cast<cuuint64_t>(grid[0])};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(head_dim) * 2, row, row * grid[2],
                                 row * grid[2] * grid[1]};
  const cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(win[2]), static_cast<cuuint32_t>(win[1]),
                             static_cast<cuuint32_t>(frames)};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool device_is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  return major == 10 && minor == 3;
}

h3_status from_cuda(cudaError_t e) { return e == cudaSuccess ? H3_OK : H3_ERR_CUDA; }

void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  The name of a __device__ array in
// host code is only a host-side stand-in, so the real address is looked up once per device with
// that device current; nullptr on failure.
void* noalloc_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

std::atomic<uint64_t> g_wait_limit_ns{0};  // 0: the default
std::atomic<int32_t> g_stall_after{-1};    // negative: never

}  // namespace

namespace h3 {
uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v == 0 ? kDefaultWaitLimitNs : v;
}
uint32_t stall_after_tiles() {
  const int32_t v = g_stall_after.load(std::memory_order_relaxed);
  return v < 0 ? 0xffffffffu : static_cast<uint32_t>(v);
}
}  // namespace h3

extern "C" {

int32_t h3_version(void) { return 100; }

uint64_t h3_set_wait_limit_ns(uint64_t nanoseconds) {
  const uint64_t prev = h3::wait_limit_ns();
  g_wait_limit_ns.store(nanoseconds, std::memory_order_relaxed);
  return prev;
}

int32_t h3_debug_stall_loads(int32_t tiles) {
  return g_stall_after.exchange(tiles < 0 ? -1 : tiles, std::memory_order_relaxed);
}

const char* h3_status_string(h3_status s) {
  switch (s) {
    case H3_OK: return "ok";
    case H3_ERR_NULL: return "a required pointer is NULL";
    case H3_ERR_INVALID_ARG: return "a size or scalar argument is out of range";
    case H3_ERR_BAD_CU_SEQLENS:
      return "cu_seqlens is not 0-based and non-decreasing within capacity, or a segment exceeds "
             "max_seqlen";
    case H3_ERR_UNSUPPORTED: return "unsupported head_dim or device (needs sm_103a, D in {64,128})";
    case H3_ERR_WORKSPACE: return "workspace missing or too small";
    case H3_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case H3_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case H3_ERR_MISALIGNED: return "a device pointer or row size is not 16-byte aligned";
    case H3_ERR_BAD_PERM: return "a permutation entry is out of range";
    case H3_ERR_BAD_BLOCK_INDEX: return "a selected block index is out of range";
  }
  return "unknown status";
}

h3_status h3_get_device_error(h3_stream_t stream) {
  unsigned int* p = device_error_ptr();
  if (p == nullptr) return H3_ERR_CUDA;
  unsigned int host = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&host, p, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return H3_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(unsigned int), st) != cudaSuccess) return H3_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return H3_ERR_CUDA;
  return static_cast<h3_status>(host);
}

h3_status h3_rope_apply(const void* q_in, void* q_out, const void* k_in, void* k_out,
                        int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                        const float* pos, const uint8_t* tag, const int32_t* cu_requests,
                        int32_t num_requests, const float* start_frames,
                        const h3_rope_cfg* cfg, h3_stream_t stream) {
  if (q_in == nullptr || q_out == nullptr || pos == nullptr || tag == nullptr) return H3_ERR_NULL;
  if ((k_in == nullptr) != (k_out == nullptr)) return H3_ERR_NULL;
  if (num_tokens < 0 || num_heads <= 0) return H3_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (cu_requests != nullptr && num_requests <= 0) return H3_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_tokens) * num_heads * head_dim / 8 > INT32_MAX)
    return H3_ERR_INVALID_ARG;
  if (!aligned16(q_in) || !aligned16(q_out) || (k_in && (!aligned16(k_in) || !aligned16(k_out))))
    return H3_ERR_MISALIGNED;

  h3_rope_cfg c{};
  if (cfg != nullptr) c = *cfg;
  const double base_t = c.base_text > 0 ? c.base_text : 10000.0;
  const double base_v = c.base_video > 0 ? c.base_video : 10000.0;
  const double base_a = c.base_audio > 0 ? c.base_audio : 10000.0;
  int dt = c.video_dims_t, dh = c.video_dims_h, dw = c.video_dims_w;
  if (dt == 0 && dh == 0 && dw == 0) {
    dt = head_dim / 2;
    dh = head_dim / 4;
    dw = head_dim / 4;
  }
  if (dt < 0 || dh < 0 || dw < 0 || dt + dh + dw != head_dim || (dt | dh | dw) & 1)
    return H3_ERR_INVALID_ARG;

  // Frequency ladders, fp64 on the host, rounded once to fp32: theta_j = base^(-2j/d).
  h3::RopeTables tab{};
  const int P = head_dim / 2;
  for (int j = 0; j < P; ++j) {
    tab.inv_text[j] = static_cast<float>(std::pow(base_t, -2.0 * j / head_dim));
    tab.inv_audio[j] = static_cast<float>(std::pow(base_a, -2.0 * j / head_dim));
    int axis, jl, d;
    if (j < dt / 2) { axis = 0; jl = j; d = dt; }
    else if (j < (dt + dh) / 2) { axis = 1; jl = j - dt / 2; d = dh; }
    else { axis = 2; jl = j - (dt + dh) / 2; d = dw; }
    tab.video_axis[j] = static_cast<uint8_t>(axis);
    tab.inv_video[j] = static_cast<float>(std::pow(base_v, -2.0 * jl / d));
  }
  tab.audio_hz = c.audio_hz > 0 ? c.audio_hz : 40.f;
  tab.video_fps = c.video_fps > 0 ? c.video_fps : 24.f;

  const int nreq = cu_requests ? num_requests : 1;
  return from_cuda(h3::launch_rope(q_in, q_out, k_in, k_out, num_tokens, num_heads, head_dim, pos,
                                   tag, cu_requests, nreq, start_frames, tab,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t h3_varlen_attn_workspace_size(int32_t num_segments, int32_t num_heads, int32_t max_seqlen,
                                     int32_t head_dim) {
  (void)num_heads;
  if (num_segments <= 0) return 0;
  return h3::attn_workspace_bytes(num_segments, max_seqlen, head_dim);
}

h3_status h3_varlen_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* cu_seqlens, int32_t num_segments, int32_t max_seqlen,
                             int32_t capacity, int32_t num_heads, int32_t head_dim,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             h3_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || cu_seqlens == nullptr)
    return H3_ERR_NULL;
  if (num_segments < 0 || num_segments > 65535 || max_seqlen < 0 || capacity < 0 ||
      num_heads <= 0 || num_heads > 65535)
    return H3_ERR_INVALID_ARG;
  if (max_seqlen > capacity) return H3_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!(softmax_scale <= 0.f || std::isfinite(softmax_scale))) return H3_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return H3_ERR_MISALIGNED;
  // the plan is required; the split area after it is used when the workspace holds it
  const size_t need = num_segments > 0 ? h3::attn_plan_bytes(num_segments) : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return H3_ERR_WORKSPACE;
  if (workspace != nullptr && !aligned16(workspace)) return H3_ERR_MISALIGNED;
  // work items are counted in 32 bits: (capacity / 256 + segments) * heads must fit
  if ((static_cast<int64_t>(capacity) / 256 + num_segments) * num_heads > INT32_MAX)
    return H3_ERR_INVALID_ARG;
  if (num_segments == 0 || max_seqlen == 0 || capacity == 0) return H3_OK;
  if (!device_is_sm103()) return H3_ERR_UNSUPPORTED;

  h3::AttnArgs a{};
  if (!make_qkv_map(&a.tmap_q, q, capacity, num_heads, head_dim) ||
      !make_qkv_map(&a.tmap_k, k, capacity, num_heads, head_dim) ||
      !make_qkv_map(&a.tmap_v, v, capacity, num_heads, head_dim))
    return H3_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.cu_seqlens = cu_seqlens;
  a.num_segments = num_segments;
  a.max_seqlen = max_seqlen;
  a.capacity = capacity;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(head_dim));
  a.workspace = workspace;
  if (max_seqlen >= h3::kSplitMinSeqlen && workspace_bytes >= need + h3::attn_split_bytes(head_dim))
    a.split_area = static_cast<uint8_t*>(workspace) + need;
  a.err = device_error_ptr();
  a.wait_limit_ns = h3::wait_limit_ns();
  a.stall_after_tiles = h3::stall_after_tiles();
  if (a.err == nullptr) return H3_ERR_CUDA;
  return from_cuda(h3::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

h3_status h3_varlen_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                     float* lse, const int32_t* cu_seqlens, int32_t num_segments,
                                     int32_t max_seqlen, int32_t capacity, int32_t num_heads,
                                     int32_t head_dim, float softmax_scale, h3_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || cu_seqlens == nullptr)
    return H3_ERR_NULL;
  if (num_segments < 0 || num_segments > 65535 || max_seqlen < 0 || capacity < 0 ||
      num_heads <= 0 || num_heads > 65535)
    return H3_ERR_INVALID_ARG;
  if (max_seqlen > capacity) return H3_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (!(softmax_scale <= 0.f || std::isfinite(softmax_scale))) return H3_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return H3_ERR_MISALIGNED;
  // the plan must fit the fixed array: refuse more segments than it was sized for
  if (num_segments > H3_NOALLOC_MAX_SEGMENTS ||
      h3::attn_plan_bytes(num_segments) > static_cast<size_t>(kNoallocScratchBytes))
    return H3_ERR_WORKSPACE;
  if ((static_cast<int64_t>(capacity) / 256 + num_segments) * num_heads > INT32_MAX)
    return H3_ERR_INVALID_ARG;
  if (num_segments == 0 || max_seqlen == 0 || capacity == 0) return H3_OK;
  if (!device_is_sm103()) return H3_ERR_UNSUPPORTED;

  void* scratch = noalloc_scratch_ptr();
  if (scratch == nullptr) return H3_ERR_CUDA;
  h3::AttnArgs a{};
  if (!make_qkv_map(&a.tmap_q, q, capacity, num_heads, head_dim) ||
      !make_qkv_map(&a.tmap_k, k, capacity, num_heads, head_dim) ||
      !make_qkv_map(&a.tmap_v, v, capacity, num_heads, head_dim))
    return H3_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.cu_seqlens = cu_seqlens;
  a.num_segments = num_segments;
  a.max_seqlen = max_seqlen;
  a.capacity = capacity;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(head_dim));
  a.workspace = scratch;  // the plan kernel rewrites every word the attention kernel reads
  a.err = device_error_ptr();
  a.wait_limit_ns = h3::wait_limit_ns();
  a.stall_after_tiles = h3::stall_after_tiles();
  if (a.err == nullptr) return H3_ERR_CUDA;
  return from_cuda(h3::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

h3_status h3_window_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                             int32_t num_heads, int32_t head_dim, float softmax_scale,
                             h3_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || grid == nullptr ||
      win == nullptr || shift == nullptr)
    return H3_ERR_NULL;
  const int32_t nwin = h3_window_count(grid, win, shift);
  if (nwin < 0 || num_heads <= 0) return H3_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return H3_ERR_UNSUPPORTED;
  // a 128-row tile is whole frames of a window, and a window is at most two tiles
  const int per_frame = win[1] * win[2];
  if (per_frame > 128 || 128 % per_frame != 0 || win[0] * per_frame > 256 || win[1] > 256 ||
      win[2] > 256)
    return H3_ERR_UNSUPPORTED;
  if (!(softmax_scale <= 0.f || std::isfinite(softmax_scale))) return H3_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(grid[0]) * grid[1] * grid[2];
  if (n > INT32_MAX / 2 || static_cast<int64_t>(nwin) * num_heads > INT32_MAX)
    return H3_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return H3_ERR_MISALIGNED;
  if (!device_is_sm103()) return H3_ERR_UNSUPPORTED;

  h3::AttnArgs a{};
  a.mode = h3::kAttnModeWindow;
  const int frames = 128 / per_frame;
  for (int ax = 0; ax < 3; ++ax) {
    a.wg.L[ax] = grid[ax];
    a.wg.w[ax] = win[ax];
    a.wg.s[ax] = shift[ax];
    a.wg.nwin[ax] = (grid[ax] + shift[ax] + win[ax] - 1) / win[ax];
  }
  a.wg.frames_per_tile = frames;
  if (!make_window_map(&a.tmap_q, q, grid, win, frames, num_heads, head_dim) ||
      !make_window_map(&a.tmap_k, k, grid, win, frames, num_heads, head_dim) ||
      !make_window_map(&a.tmap_v, v, grid, win, frames, num_heads, head_dim))
    return H3_ERR_CUDA;
  // half-height boxes for edge windows with at most half their rows along H inside the grid
  a.wg.half_h = win[1] % 2 == 0 ? 1 : 0;
  if (a.wg.half_h) {
    const int32_t half_win[3] = {win[0], win[1] / 2, win[2]};
    if (!make_window_map(&a.tmap_q2, q, grid, half_win, 2 * frames, num_heads, head_dim) ||
        !make_window_map(&a.tmap_k2, k, grid, half_win, 2 * frames, num_heads, head_dim) ||
        !make_window_map(&a.tmap_v2, v, grid, half_win, 2 * frames, num_heads, head_dim))
      return H3_ERR_CUDA;
  }
  a.o = o;
  a.lse = lse;
  a.capacity = static_cast<int>(n);  // LSE row stride: [heads, T*H*W]
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(head_dim));
  a.err = device_error_ptr();
  a.wait_limit_ns = h3::wait_limit_ns();
  a.stall_after_tiles = h3::stall_after_tiles();
  if (a.err == nullptr) return H3_ERR_CUDA;
  return from_cuda(h3::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

// ---- continuation window ------------------------------------------------------------------------

h3_status h3_continuation_make_plan(const h3_continuation_cfg* c, h3_continuation_plan* p) {
  if (c == nullptr || p == nullptr) return H3_ERR_NULL;
  if (c->text_rows < 0 || c->clip_video_frames < 0 || c->clip_audio_rows < 0 || c->frame_h <= 0 ||
      c->frame_w <= 0 || c->new_video_frames < 0 || c->new_audio_rows < 0 || c->tail_frames < 0 ||
      c->frames_per_latent <= 0)
    return H3_ERR_INVALID_ARG;
  const int64_t g0 = static_cast<int64_t>(c->clip_video_frames) - c->tail_frames;
  if (g0 < 0 || c->new_video_frames < c->tail_frames) return H3_ERR_INVALID_ARG;
  const int64_t s = g0 * c->frames_per_latent;
  if (s > INT32_MAX / 40) return H3_ERR_INVALID_ARG;
  const int64_t cut = std::min<int64_t>(s * 40 / 24, c->clip_audio_rows);  // floor(s * 40 / 24)
  const int64_t ref_audio = c->clip_audio_rows - cut;
  if (c->new_audio_rows < ref_audio) return H3_ERR_INVALID_ARG;
  const int64_t hw = static_cast<int64_t>(c->frame_h) * c->frame_w;
  const int64_t rows[5] = {c->text_rows, ref_audio, c->tail_frames * hw, c->new_audio_rows,
                           c->new_video_frames * hw};
  int64_t off = 0;
  for (int k = 0; k < 5; ++k) {
    p->group_offset[k] = static_cast<int32_t>(off);
    off += rows[k];
    if (off > INT32_MAX) return H3_ERR_INVALID_ARG;
    p->group_rows[k] = static_cast<int32_t>(rows[k]);
  }
  p->group_offset[5] = static_cast<int32_t>(off);
  p->num_rows = static_cast<int32_t>(off);
  p->tail_start = static_cast<int32_t>(g0);
  p->start_frame = static_cast<int32_t>(s);
  p->audio_cut = static_cast<int32_t>(cut);
  p->keep_video_from = c->tail_frames;
  p->keep_audio_from = static_cast<int32_t>(ref_audio);
  if (g0 + c->new_video_frames > INT32_MAX || cut + c->new_audio_rows > INT32_MAX)
    return H3_ERR_INVALID_ARG;
  p->out_video_frames = static_cast<int32_t>(g0 + c->new_video_frames);
  p->out_audio_rows = static_cast<int32_t>(cut + c->new_audio_rows);
  return H3_OK;
}

h3_status h3_continuation_pack(const h3_continuation_cfg* cfg, const void* text,
                               const void* clip_video, const void* clip_audio,
                               const void* new_video, const void* new_audio, int32_t row_bytes,
                               void* rows, float* pos, uint8_t* tag, uint8_t* target,
                               h3_stream_t stream) {
  if (cfg == nullptr || rows == nullptr || pos == nullptr || tag == nullptr || target == nullptr)
    return H3_ERR_NULL;
  h3_continuation_plan p;
  const h3_status st = h3_continuation_make_plan(cfg, &p);
  if (st != H3_OK) return st;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return H3_ERR_INVALID_ARG;
  const void* src[5] = {text, clip_audio, clip_video, new_audio, new_video};
  for (int k = 0; k < 5; ++k) {
    if (p.group_rows[k] > 0 && src[k] == nullptr) return H3_ERR_NULL;
    if (src[k] != nullptr && !aligned16(src[k])) return H3_ERR_MISALIGNED;
  }
  if (static_cast<int64_t>(p.num_rows) * row_bytes / 16 > INT64_MAX / 4) return H3_ERR_INVALID_ARG;
  if (!aligned16(rows) || (reinterpret_cast<uintptr_t>(pos) & 3u)) return H3_ERR_MISALIGNED;
  const int64_t hw = static_cast<int64_t>(cfg->frame_h) * cfg->frame_w;
  const int64_t first[5] = {0, p.audio_cut, static_cast<int64_t>(p.tail_start) * hw, 0, 0};
  h3::ContinuationGeom g;
  for (int k = 0; k < 5; ++k) g.offset[k] = p.group_offset[k];
  g.num_rows = p.num_rows;
  g.frame_h = cfg->frame_h;
  g.frame_w = cfg->frame_w;
  return from_cuda(h3::launch_continuation_pack(g, src, first, row_bytes, rows, pos, tag, target,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

h3_status h3_continuation_append(const h3_continuation_cfg* cfg, const void* new_video,
                                 const void* new_audio, int32_t row_bytes, void* clip_video,
                                 int64_t clip_video_capacity_rows, void* clip_audio,
                                 int64_t clip_audio_capacity_rows, h3_stream_t stream) {
  if (cfg == nullptr) return H3_ERR_NULL;
  h3_continuation_plan p;
  const h3_status st = h3_continuation_make_plan(cfg, &p);
  if (st != H3_OK) return st;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return H3_ERR_INVALID_ARG;
  const int64_t hw = static_cast<int64_t>(cfg->frame_h) * cfg->frame_w;
  const int64_t v_rows = (static_cast<int64_t>(cfg->new_video_frames) - p.keep_video_from) * hw;
  const int64_t a_rows = static_cast<int64_t>(cfg->new_audio_rows) - p.keep_audio_from;
  if ((v_rows > 0 && (new_video == nullptr || clip_video == nullptr)) ||
      (a_rows > 0 && (new_audio == nullptr || clip_audio == nullptr)))
    return H3_ERR_NULL;
  if (static_cast<int64_t>(p.out_video_frames) * hw > clip_video_capacity_rows && v_rows > 0)
    return H3_ERR_INVALID_ARG;
  if (p.out_audio_rows > clip_audio_capacity_rows && a_rows > 0) return H3_ERR_INVALID_ARG;
  for (const void* ptr : {new_video, new_audio, static_cast<const void*>(clip_video),
                          static_cast<const void*>(clip_audio)})
    if (ptr != nullptr && !aligned16(ptr)) return H3_ERR_MISALIGNED;
  const char* nv = static_cast<const char*>(new_video);
  const char* na = static_cast<const char*>(new_audio);
  char* cv = static_cast<char*>(clip_video);
  char* ca = static_cast<char*>(clip_audio);
  const void* src[2] = {v_rows > 0 ? nv + p.keep_video_from * hw * row_bytes : nullptr,
                        a_rows > 0 ? na + static_cast<int64_t>(p.keep_audio_from) * row_bytes : nullptr};
  void* dst[2] = {v_rows > 0 ? cv + cfg->clip_video_frames * hw * row_bytes : nullptr,
                  a_rows > 0 ? ca + static_cast<int64_t>(cfg->clip_audio_rows) * row_bytes : nullptr};
  const int64_t bytes[2] = {v_rows > 0 ? v_rows * row_bytes : 0, a_rows > 0 ? a_rows * row_bytes : 0};
  return from_cuda(h3::launch_copy_ranges(src, dst, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

h3_status h3_masked_row_update(void* dst, const void* src, const uint8_t* mask, int32_t num_rows,
                               int32_t row_bytes, h3_stream_t stream) {
  if (num_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return H3_ERR_INVALID_ARG;
  if (num_rows == 0) return H3_OK;
  if (dst == nullptr || src == nullptr || mask == nullptr) return H3_ERR_NULL;
  if (!aligned16(dst) || !aligned16(src)) return H3_ERR_MISALIGNED;
  return from_cuda(h3::launch_masked_row_update(dst, src, mask, num_rows, row_bytes,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

// ---- VSA ----------------------------------------------------------------------------------------

int32_t h3_vsa_block_count(const int32_t grid[3], const int32_t block[3]) {
  if (grid == nullptr || block == nullptr) return -1;
  int64_t n = 1;
  for (int a = 0; a < 3; ++a) {
    if (grid[a] <= 0 || block[a] <= 0) return -1;
    n *= (static_cast<int64_t>(grid[a]) + block[a] - 1) / block[a];
  }
  return n > INT32_MAX ? -1 : static_cast<int32_t>(n);
}

namespace {

// Shared checks of the VSA calls: a 64-token block (one half of a 128-row tile), a grid whose
// rows and blocks fit the kernels' int32 indexing.
h3_status vsa_geometry(const int32_t grid[3], const int32_t block[3], int32_t num_heads,
                       int32_t head_dim, h3::VsaGeom* g) {
  const int32_t nblk = h3_vsa_block_count(grid, block);
  if (nblk < 0 || num_heads <= 0) return H3_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return H3_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(block[0]) * block[1] * block[2] != 64) return H3_ERR_UNSUPPORTED;
  const int64_t n = static_cast<int64_t>(grid[0]) * grid[1] * grid[2];
  if (n > INT32_MAX / 2 || static_cast<int64_t>(nblk) * num_heads > INT32_MAX / 4)
    return H3_ERR_INVALID_ARG;
  for (int a = 0; a < 3; ++a) {
    g->L[a] = grid[a];
    g->b[a] = block[a];
    g->nb[a] = (grid[a] + block[a] - 1) / block[a];
  }
  return H3_OK;
}

}  // namespace

size_t h3_vsa_select_workspace_size(const int32_t grid[3], const int32_t block[3],
                                    int32_t num_heads, int32_t head_dim) {
  h3::VsaGeom g;
  if (vsa_geometry(grid, block, num_heads, head_dim, &g) != H3_OK) return 0;
  return h3::vsa_pool_bytes(g.nb[0] * g.nb[1] * g.nb[2], num_heads, head_dim);
}

h3_status h3_vsa_select(const void* q, const void* k, const int32_t grid[3],
                        const int32_t block[3], int32_t num_heads, int32_t head_dim,
                        int32_t topk, float softmax_scale, float* scores, int32_t* block_idx,
                        void* workspace, size_t workspace_bytes, h3_stream_t stream) {
  if (q == nullptr || k == nullptr || grid == nullptr || block == nullptr || scores == nullptr ||
      block_idx == nullptr)
    return H3_ERR_NULL;
  h3::VsaGeom g;
  const h3_status st = vsa_geometry(grid, block, num_heads, head_dim, &g);
  if (st != H3_OK) return st;
  const int64_t nblk = static_cast<int64_t>(g.nb[0]) * g.nb[1] * g.nb[2];
  if (topk < 1 || topk > nblk) return H3_ERR_INVALID_ARG;
  if (nblk * nblk * num_heads > (static_cast<int64_t>(1) << 40)) return H3_ERR_INVALID_ARG;
  if (!(softmax_scale <= 0.f || std::isfinite(softmax_scale))) return H3_ERR_INVALID_ARG;
  if (workspace == nullptr ||
      workspace_bytes < h3::vsa_pool_bytes(static_cast<int>(nblk), num_heads, head_dim))
    return H3_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(block_idx) & 3u))
    return H3_ERR_MISALIGNED;
  if (!device_is_sm103()) return H3_ERR_UNSUPPORTED;
  const float scale =
      softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(head_dim));
  return from_cuda(h3::launch_vsa_select(q, k, g, num_heads, head_dim, topk, scale, scores,
                                         block_idx, workspace,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

size_t h3_vsa_attn_workspace_size(const int32_t grid[3], const int32_t block[3],
                                  int32_t num_heads, int32_t topk) {
  h3::VsaGeom g;
  if (grid == nullptr || block == nullptr ||
      vsa_geometry(grid, block, num_heads, 128, &g) != H3_OK)
    return 0;
  const int nblk = g.nb[0] * g.nb[1] * g.nb[2];
  if (topk < 1 || topk > nblk) return 0;
  return h3::vsa_schedule_bytes(nblk, num_heads, topk);
}

h3_status h3_vsa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t grid[3], const int32_t block[3], int32_t num_heads,
                          int32_t head_dim, const int32_t* block_idx, int32_t topk,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          h3_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || grid == nullptr ||
      block == nullptr || block_idx == nullptr)
    return H3_ERR_NULL;
  h3::VsaGeom g;
  const h3_status st = vsa_geometry(grid, block, num_heads, head_dim, &g);
  if (st != H3_OK) return st;
  const int64_t nblk = static_cast<int64_t>(g.nb[0]) * g.nb[1] * g.nb[2];
  if (topk < 1 || topk > nblk || nblk > static_cast<int64_t>(h3::kVsaBlockMask))
    return H3_ERR_INVALID_ARG;
  if (!(softmax_scale <= 0.f || std::isfinite(softmax_scale))) return H3_ERR_INVALID_ARG;
  const size_t need = h3::vsa_schedule_bytes(static_cast<int>(nblk), num_heads, topk);
  if (workspace == nullptr || workspace_bytes < need) return H3_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (reinterpret_cast<uintptr_t>(block_idx) & 3u))
    return H3_ERR_MISALIGNED;
  if (!device_is_sm103()) return H3_ERR_UNSUPPORTED;
  unsigned int* err = device_error_ptr();
  if (err == nullptr) return H3_ERR_CUDA;

  h3::AttnArgs a{};
  a.mode = h3::kAttnModeVsa;
  for (int ax = 0; ax < 3; ++ax) {
    a.wg.L[ax] = grid[ax];
    a.wg.w[ax] = block[ax];
    a.wg.s[ax] = 0;
    a.wg.nwin[ax] = g.nb[ax];
  }
  a.wg.topk = topk;
  const size_t pairs = static_cast<size_t>(num_heads) * h3::vsa_pairs(static_cast<int>(nblk));
  a.vsa_steps = static_cast<const uint2*>(workspace);
  a.vsa_counts = reinterpret_cast<const int2*>(static_cast<const uint8_t*>(workspace) +
                                              (pairs * topk * 8 + 255) / 256 * 256);
  // one block (bw x bh x bt = 64 rows) per box
  if (!make_window_map(&a.tmap_q, q, grid, block, block[0], num_heads, head_dim) ||
      !make_window_map(&a.tmap_k, k, grid, block, block[0], num_heads, head_dim) ||
      !make_window_map(&a.tmap_v, v, grid, block, block[0], num_heads, head_dim))
    return H3_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.capacity = grid[0] * grid[1] * grid[2];  // LSE row stride: [heads, T*H*W]
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(head_dim));
  a.err = err;
  a.wait_limit_ns = h3::wait_limit_ns();
  a.stall_after_tiles = h3::stall_after_tiles();
  // the pairs' key/value schedule, then the attention that follows it (same stream)
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t ce = h3::launch_vsa_schedule(block_idx, static_cast<int>(nblk), num_heads,
                                                 topk, workspace, err, cs);
  if (ce != cudaSuccess) return from_cuda(ce);
  return from_cuda(h3::launch_attn_fwd(a, cs));
}

int32_t h3_window_count(const int32_t grid[3], const int32_t win[3], const int32_t shift[3]) {
  if (grid == nullptr || win == nullptr || shift == nullptr) return -1;
  int64_t n = 1;
  for (int a = 0; a < 3; ++a) {
    if (grid[a] <= 0 || win[a] <= 0 || shift[a] < 0 || shift[a] >= win[a]) return -1;
    n *= (static_cast<int64_t>(grid[a]) + shift[a] + win[a] - 1) / win[a];
  }
  return n > INT32_MAX ? -1 : static_cast<int32_t>(n);
}

h3_status h3_window_pack(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                         int32_t* perm, int32_t* cu_seqlens, const void* const* src,
                         void* const* dst, int32_t num_tensors, int32_t row_bytes,
                         h3_stream_t stream) {
  if (grid == nullptr || win == nullptr || shift == nullptr || perm == nullptr ||
      cu_seqlens == nullptr)
    return H3_ERR_NULL;
  if (num_tensors < 0 || num_tensors > h3::kMaxPackTensors) return H3_ERR_INVALID_ARG;
  if (num_tensors > 0 && (src == nullptr || dst == nullptr)) return H3_ERR_NULL;
  const int32_t nwin = h3_window_count(grid, win, shift);
  if (nwin < 0) return H3_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(grid[0]) * grid[1] * grid[2];
  if (n > INT32_MAX / 2) return H3_ERR_INVALID_ARG;
  h3::PackPtrs ptrs{};
  if (num_tensors > 0) {
    if (row_bytes <= 0 || (row_bytes & 15)) return H3_ERR_MISALIGNED;
    for (int i = 0; i < num_tensors; ++i) {
      if (src[i] == nullptr || dst[i] == nullptr) return H3_ERR_NULL;
      if (!aligned16(src[i]) || !aligned16(dst[i])) return H3_ERR_MISALIGNED;
      ptrs.src[i] = src[i];
      ptrs.dst[i] = dst[i];
    }
  }
  h3::WindowGeom g{};
  for (int a = 0; a < 3; ++a) {
    g.L[a] = grid[a];
    g.w[a] = win[a];
    g.s[a] = shift[a];
    g.nwin[a] = (grid[a] + shift[a] + win[a] - 1) / win[a];
  }
  return from_cuda(h3::launch_window_pack(g, perm, cu_seqlens, ptrs, num_tensors, row_bytes,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

h3_status h3_window_unpack(const int32_t* perm, int32_t num_tokens, const void* src, void* dst,
                           int32_t row_bytes, h3_stream_t stream) {
  if (perm == nullptr || src == nullptr || dst == nullptr) return H3_ERR_NULL;
  if (num_tokens < 0) return H3_ERR_INVALID_ARG;
  if (row_bytes <= 0 || (row_bytes & 15)) return H3_ERR_MISALIGNED;
  if (!aligned16(src) || !aligned16(dst)) return H3_ERR_MISALIGNED;
  unsigned int* err = device_error_ptr();
  if (err == nullptr) return H3_ERR_CUDA;
  return from_cuda(h3::launch_window_unpack(perm, num_tokens, src, dst, row_bytes, err,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
