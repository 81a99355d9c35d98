// Softmax attention forward for sm_103a: TMA + tcgen05 + TMEM, in three variants of one kernel
// template (the warp roles, rings, barriers and TMEM plan below are shared):
//   kModePacked  block-diagonal attention over the cu_seqlens segments of a packed sequence;
//   kModeWindow  3D (shifted) window attention read and written in place on a (T, H, W) grid:
//                a 128-row tile is one 5-D TMA box of whole window frames, edge windows masked;
//   kModeVsa     block-sparse video attention: a tile holds two 64-token query blocks, each
//                attending to its own selected key blocks, stacked in every key/value tile.
// The description below is that of the packed variant; the others differ where noted in code.
//
// [H3-vLLM] "Joint audio/video generation in production: MiniMax-H3 and vLLM-Omni", sec. 3:
// cu_seqlens holds the offsets of the sub-sequences packed into one sequence; a query of
// sub-sequence g softmax-normalises over the keys of g only (no causal mask: the worked
// example's token 15 sees keys 10..29).  Sec. 6: rows past the valid length never take part.
//
// Work item: two 128-row query tiles (256 rows) of one segment and one head; both tiles stream
// the same key/value tiles, so each K/V tile staged in shared memory feeds twice the
// tensor-core work.  No tile crosses a segment boundary: query and key/value tiles start at the
// segment's first row (TMA boxes may start at any row), so only the segment's LAST key tile can
// overhang.  On that tile the overhanging key columns are masked to -inf by select, and the
// overhanging value rows are zeroed in shared memory before the PV product (0 * NaN would
// otherwise leak a neighbour's or a pad row's NaN).  Overhanging query rows are never stored.
//
// Scheduling: a one-CTA plan kernel validates cu_seqlens, orders the segments longest first
// (up to kSortMax segments; beyond that in given order) and writes the exclusive prefix of work
// items per segment into the caller's workspace.  CTA c takes items c, c + G, c + 2G, ... (G =
// grid size); its TMA warp decodes each item and hands it to the other roles through a 2-slot
// ring in shared memory.  For short segments (max_seqlen <= kPersistMaxSeqlen) the grid is one
// CTA per SM and each CTA loops over items: the K/V ring, the Q reload (after the item's last
// QK^T) and the epilogue (before the next item's first PV) overlap consecutive items, which pays
// for 3D windows of a few hundred rows.  For long segments the grid has one CTA per item (set
// up per item costs little against hundreds of key tiles, and measured faster there).  Items of
// one segment are numbered head-major, so the CTAs working at one time share a head's K/V in L2.
//
// Warp roles (384 threads = 3 warpgroups; registers moved to the softmax warpgroups with
// setmaxnreg: 200 each for warpgroups 0 and 1, 104 for warpgroup 2):
//   warps 0-3 / 4-7  softmax of query tile 0 / 1: thread r owns query row r = TMEM lane r and
//              reads its full row of S = Q K^T (128 fp32) with tcgen05.ld, so the row max and
//              row sum need no shuffles.  Running max and sum stay in fp32; P is written back to
//              TMEM over S as bf16 (the A operand of the PV product); O is rescaled in TMEM only
//              when the running max grows by more than 2^8; the epilogue normalises O and
//              stores it (and the LSE).
//   warp 8     scheduler + TMA producer: Q tiles once per item, then K and V tiles through
//              rings that run on across items (at D = 128: 3 K / 2 V stages for packed
//              segments and VSA, 2 K / 3 V for windows).
//   warp 9     MMA issuer (one thread).  Order per key tile j:
//                PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
//              so while softmax 0 works on S0_{j+1} the tensor core runs PV1_j and S1_{j+1},
//              and vice versa (ping-pong).  Because S_t,{j+1} is issued after PV_t,j, seeing
//              S_t,{j+1} complete also means O_t is stable for an in-place rescale.  In the
//              packed and window variants the softmax publishes P over the first 64 keys on
//              its own barrier, and PV_t,j runs as two halves of 64 keys, the first while the
//              softmax still exponentiates the second half of the row.
//   warp 10    VSA only: TMA producer of the V tiles (the K tiles stay with warp 8).
//   warp 11    idle (it completes warpgroup 2).
// TMEM (512 columns): O0 [0,128), O1 [128,256), S0/P0 [256,384), S1/P1 [384,512).
//
// Barrier phases run on across items: every role counts its own completions and derives each
// wait's parity from them; no waiter can fall more than one phase behind its barrier.
#include <cuda_bf16.h>

#include <atomic>

#include <type_traits>
#include <utility>

#include "h3_internal.h"
#include "sm103_ptx.cuh"

namespace h3 {
namespace {

constexpr int kBlockM = 128;          // query rows per tile
constexpr int kBlockN = 128;          // keys per tile
constexpr int kTilesPerItem = 2;      // query tiles per work item
constexpr int kRowsPerItem = kTilesPerItem * kBlockM;
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 200;  // 128 * (200 + 200 + 104) = 384 * 168 registers at launch
constexpr int kRegsOther = 104;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;              // O of tile t at kColO + 128 t
constexpr int kColS = 256;            // S / P of tile t at kColS + 128 t
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the running max grows by > 2^8
constexpr int kPlanThreads = 1024;
constexpr int kSortMax = 256;         // segments ordered longest-first up to this count
constexpr int kWsHeader = kAttnWsHeaderWords;  // workspace words: (spare), total items, 2 spare
constexpr int kPersistMaxSeqlen = 2048;  // loop over items per CTA up to this segment length
constexpr int kPersistMaxWaves = 8;      // ... or when the job has at most this many waves of items

static_assert(kDefaultWaitLimitNs == kWaitLimitNs, "host and device default wait limits agree");

constexpr int kModePacked = kAttnModePacked;  // kernel variants (see h3_internal.h)
constexpr int kModeWindow = kAttnModeWindow;
constexpr int kModeVsa = kAttnModeVsa;
constexpr int kVsaBlockRows = 64;  // rows of one VSA block = half a 128-row tile


// Packed segments: the key/value tiles [kv0, kv0 + nkv) an item covers (all of its segment's,
// unless the item is a chunk of a split one) and the split: (chunk << 16 | chunks), 0 for a
// whole item; group = the split item's first entry in the split area.
struct PackedChunk {
  int kv0, split, group;
};

struct WorkDesc {
  int seg_start;  // packed: first row of the segment
  int seg_len;    // packed: rows of the segment; window: 1; < 0: no more work
  int head;
  int q0;         // packed: first query row of the item
  int box[3];     // window: grid (t, h, w) of the first valid tile's box origin (may be < 0)
  int ntiles;     // window / VSA: query tiles of the item (1 or 2)
  int nkv;        // window / VSA: key/value steps of the item (VSA: the larger tile's)
  int nkv_t[2];   // VSA: key/value steps of each query tile
  int nsh_t[2];   // VSA: key blocks both query blocks of the tile selected
  int hbox;       // window: box rows along H (the window's, or half of it for an edge window)
  int fpt;        // window: frames per 128-row tile (128 / (hbox * window W))
  union {
    uint32_t mask[2][4];  // window: rows of each tile that lie inside the grid (= inside the window)
    PackedChunk pk;       // packed: the item's key range and split
  };
};

struct ItemShape {
  bool has1;          // second query tile present
  int nkv;            // key/value tiles
  int kv_last_valid;  // keys in the last key tile (packed; 128 for windows, which use masks)
};

template <int kMode>
__device__ __forceinline__ ItemShape shape_of(const WorkDesc& d) {
  if (kMode != kModePacked) return ItemShape{d.ntiles == 2, d.nkv, kBlockN};
  // a chunk of a split item covers key tiles [kv0, kv0 + nkv); only the segment's last key tile
  // can be partial
  const int nkv_seg = (d.seg_len + kBlockN - 1) / kBlockN;
  const int last = d.pk.kv0 + d.nkv == nkv_seg ? d.seg_len - (nkv_seg - 1) * kBlockN : kBlockN;
  return ItemShape{d.q0 + kBlockM < d.seg_start + d.seg_len, d.nkv, last};
}

// 128-bit row masks as (lo, hi) 64-bit halves.
__device__ __forceinline__ void or_shifted(uint64_t& lo, uint64_t& hi, uint64_t lo_in, uint64_t hi_in,
                                           int sh) {  // (lo, hi) |= (lo_in, hi_in) << sh, sh < 128
  if (sh == 0) {
    lo |= lo_in;
    hi |= hi_in;
  } else if (sh < 64) {
    lo |= lo_in << sh;
    hi |= (hi_in << sh) | (lo_in >> (64 - sh));
  } else {
    hi |= lo_in << (sh - 64);
  }
}
__device__ __forceinline__ uint64_t low_bits(int n) {  // n in [0, 64]
  return n >= 64 ? ~0ull : ((1ull << n) - 1ull);
}

// Window item -> descriptor.  Items are numbered window-major, head fastest, so CTAs working at
// one time read neighbouring 256-byte pieces of the same token rows.  Along each axis the window's
// box starts at i * w - s (the shifted grid; may be negative) and the rows inside the grid are
// [max(0, start), min(L, start + w)): the rest of the box is zero-filled by TMA and masked.
// An edge window whose rows inside the grid along H fit in half the window (g.half_h) uses the
// half-height box, starting at its first valid row, with twice the frames per tile: the shifted
// layer's top and bottom windows then take one tile instead of two.
// The masks are built in registers: a frame mask (valid h rows x valid w run), then per tile the
// valid frames of that tile.
__device__ __forceinline__ WorkDesc decode_window(uint32_t item, const WindowAttnGeom& g,
                                                  int num_heads) {
  const int win = static_cast<int>(item / static_cast<uint32_t>(num_heads));
  WorkDesc d{};
  d.seg_len = 1;
  d.head = static_cast<int>(item % static_cast<uint32_t>(num_heads));
  const int iw = win % g.nwin[2], ih = (win / g.nwin[2]) % g.nwin[1], it = win / (g.nwin[2] * g.nwin[1]);
  const int lo_t = it * g.w[0] - g.s[0], lo_h = ih * g.w[1] - g.s[1], lo_w = iw * g.w[2] - g.s[2];
  const int vl_t = max(0, -lo_t), vh_t = min(g.w[0], g.L[0] - lo_t);
  const int vl_h = max(0, -lo_h), vh_h = min(g.w[1], g.L[1] - lo_h);
  const int vl_w = max(0, -lo_w), vh_w = min(g.w[2], g.L[2] - lo_w);
  const bool half = g.half_h && 2 * (vh_h - vl_h) <= g.w[1];
  const int h0 = half ? vl_h : 0;  // first box row along H, relative to the window
  d.hbox = half ? g.w[1] / 2 : g.w[1];
  d.fpt = half ? 2 * g.frames_per_tile : g.frames_per_tile;
  const int bt = d.fpt;
  const int tile_lo = vl_t / bt, tile_hi = (vh_t + bt - 1) / bt;
  d.ntiles = tile_hi - tile_lo;
  d.nkv = d.ntiles;
  d.box[0] = lo_t + tile_lo * bt;
  d.box[1] = lo_h + h0;
  d.box[2] = lo_w;
  // frame mask: bits fh * ww + fw for valid (fh, fw) of the box; ww <= 128, pf = hbox * ww <= 128
  const int ww = g.w[2], pf = d.hbox * g.w[2];
  uint64_t flo = 0, fhi = 0;
  const int run = vh_w - vl_w;
  const uint64_t rlo = low_bits(min(run, 64)), rhi = run > 64 ? low_bits(run - 64) : 0ull;
  for (int fh = vl_h - h0; fh < vh_h - h0; ++fh) or_shifted(flo, fhi, rlo, rhi, fh * ww + vl_w);
#pragma unroll
  for (int k = 0; k < 2; ++k) {  // ntiles <= 2: frames_per_tile * 2 covers the window's frames
    if (k >= d.ntiles) break;
    uint64_t tlo = 0, thi = 0;
    for (int ft = 0; ft < bt; ++ft) {
      const int t = (tile_lo + k) * bt + ft;  // box-local frame
      if (t >= vl_t && t < vh_t) or_shifted(tlo, thi, flo, fhi, ft * pf);
    }
    d.mask[k][0] = static_cast<uint32_t>(tlo);
    d.mask[k][1] = static_cast<uint32_t>(tlo >> 32);
    d.mask[k][2] = static_cast<uint32_t>(thi);
    d.mask[k][3] = static_cast<uint32_t>(thi >> 32);
  }
  return d;
}

// ---- VSA: blocks of 64 tokens (bt x bh x bw) cut from the grid at multiples of the block size.
// wg.w[] holds the block size, wg.nwin[] the blocks per axis, wg.topk the selected key blocks per
// query block; block b = (i_t, i_h, i_w) lexicographic.
__device__ __forceinline__ int vsa_num_blocks(const WindowAttnGeom& g) {
  return g.nwin[0] * g.nwin[1] * g.nwin[2];
}
// Grid origin (t, h, w) of block b.
__device__ __forceinline__ void vsa_block_origin(int b, const WindowAttnGeom& g, int& t0, int& h0,
                                                 int& w0) {
  w0 = (b % g.nwin[2]) * g.w[2];
  h0 = ((b / g.nwin[2]) % g.nwin[1]) * g.w[1];
  t0 = (b / (g.nwin[2] * g.nwin[1])) * g.w[0];
}
// Rows of block b inside the grid: bit (ft * bh + fh) * bw + fw of a 64-bit mask.
__device__ __forceinline__ uint64_t vsa_block_mask(int b, const WindowAttnGeom& g) {
  int t0, h0, w0;
  vsa_block_origin(b, g, t0, h0, w0);
  const int nt = min(g.w[0], g.L[0] - t0), nh = min(g.w[1], g.L[1] - h0);
  const uint64_t run = low_bits(min(g.w[2], g.L[2] - w0));
  uint64_t frame = 0, m = 0;
  for (int fh = 0; fh < nh; ++fh) frame |= run << (fh * g.w[2]);
  for (int ft = 0; ft < nt; ++ft) m |= frame << (ft * g.w[1] * g.w[2]);
  return m;
}
// Item -> descriptor: query blocks q0 .. q0 + 3 of one head (tile t holds blocks q0 + 2t and
// q0 + 2t + 1 in its two 64-row halves: pair q0 / 2 + t of the key/value schedule).  Items are
// numbered head-major: the CTAs working at one time serve one head (two at a boundary), so the
// key/value blocks they select at random stay in L2 (one head's K and V of the 32x48x84 grid
// are 66 MB), instead of every head's at once.
__device__ __forceinline__ WorkDesc decode_vsa(uint32_t item, const WindowAttnGeom& g,
                                               const int2* __restrict__ counts) {
  WorkDesc d{};
  d.seg_len = 1;
  const int nblk = vsa_num_blocks(g);
  const uint32_t quads = static_cast<uint32_t>((nblk + 3) / 4);
  d.head = static_cast<int>(item / quads);
  d.q0 = 4 * static_cast<int>(item % quads);
  d.ntiles = d.q0 + 2 < nblk ? 2 : 1;
  const int2* c = counts + static_cast<size_t>(d.head) * ((nblk + 1) / 2) + d.q0 / 2;
  const int2 c0 = __ldg(c), c1 = d.ntiles == 2 ? __ldg(c + 1) : make_int2(0, 0);
  d.nkv_t[0] = min(max(c0.x, 1), g.topk);
  d.nkv_t[1] = d.ntiles == 2 ? min(max(c1.x, 1), g.topk) : 0;
  d.nsh_t[0] = c0.y;
  d.nsh_t[1] = c1.y;
  d.nkv = max(d.nkv_t[0], d.nkv_t[1]);
  return d;
}
// Step j of pair p (head h): the two key blocks of the step and which query block uses each.
__device__ __forceinline__ uint2 vsa_step(const uint2* __restrict__ steps, int h, int p, int j,
                                          const WindowAttnGeom& g) {
  return __ldg(steps + (static_cast<size_t>(h) * ((vsa_num_blocks(g) + 1) / 2) + p) * g.topk + j);
}

__device__ __forceinline__ int checked_len(const int32_t* __restrict__ cu, int g, int capacity,
                                           int max_seqlen, unsigned int* err) {
  const int a = cu[g], b = cu[g + 1];
  if (a < 0 || b < a || b > capacity || (g == 0 && a != 0)) {
    record_error(err, kErrBadCuSeqlens);
    return 0;  // an invalid segment produces nothing
  }
  if (b - a > max_seqlen) record_error(err, kErrBadCuSeqlens);  // computed all the same
  return b - a;
}

__device__ __forceinline__ uint32_t items_of(int len, int heads) {
  return static_cast<uint32_t>((len + kRowsPerItem - 1) / kRowsPerItem) * heads;
}

// ---- Split of the last wave (packed segments) -------------------------------------------------
// With G CTAs working at a time, items [F*G, T) of T whole items (F = T / G) form a last wave that
// leaves most SMs idle when items are long (the 4,096-token request: 336 equal video items on 152
// SMs).  The plan cuts each long item of that wave into chunks of its key tiles so that the wave's
// work spreads over all G CTAs.  Each chunk writes its partial result (O normalised by its own row
// sum, fp32, and its LSE) to the split area; a merge kernel then combines the chunks of every split
// item in chunk order (so the result does not depend on which chunk finished first):
//   lse = log sum_c exp(lse_c),   o = sum_c exp(lse_c - lse) o_c.
// Split area (after the plan, 256-byte aligned): kSplitMaxEntries entries of 8 words, the list of
// split items (their first entries; plan word 0 counts them), then per entry and query tile 128
// rows of D fp32 values followed by their 128 fp32 LSEs.
constexpr int kSplitMinTiles = 8;   // split only items of at least 8 key tiles (1,024 keys)
constexpr int kSplitMaxChunks = 8;
struct SplitEntry {
  int seg_start, seg_len, head, q0, kv0, kv1, group, split;  // split = chunk << 16 | chunks
};
static_assert(sizeof(SplitEntry) == 8 * sizeof(int32_t), "split entries are 8 words");
__host__ __device__ constexpr size_t split_groups_offset() {  // first entries of the split items
  return static_cast<size_t>(kSplitMaxEntries) * sizeof(SplitEntry);
}
__host__ __device__ constexpr size_t split_partials_offset() {
  return split_groups_offset() + static_cast<size_t>(kSplitMaxEntries) * sizeof(uint32_t);
}
static_assert(split_partials_offset() % 16 == 0, "partial rows are written as 16-byte vectors");
static_assert(split_partials_offset() + static_cast<size_t>(kSplitMaxEntries) * 2 * kBlockM * 129 *
                      sizeof(float) == attn_split_bytes(128),
              "split area layout agrees with its size");

// Merge of split items.  Work unit (group, t, z): rows [16 z, 16 z + 16) of query tile t of the
// split item whose first entry is the group's; the CTAs of a small fixed grid take the units in
// turn.  Chunks are combined in chunk order.  Memory-bound and short: the partials were written
// moments before and are read back from L2; every chunk's loads of a unit are issued together.
constexpr int kMergeThreads = 256;
constexpr int kMergeRows = 16;  // rows per unit: 16 rows x D / 8 column groups = 256 threads at D = 128
constexpr int kMergeUnitsPerGroup = 2 * (kBlockM / kMergeRows);
template <int D>
__global__ void __launch_bounds__(kMergeThreads)
attn_merge_kernel(const uint32_t* __restrict__ ws, const uint8_t* __restrict__ split_area,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int num_heads,
                  int capacity, const unsigned int* err) {
  __shared__ float s_w[kMergeRows][kSplitMaxChunks];  // per row: chunk weights exp(lse_c - lse)
  __shared__ float s_lse[kMergeRows];
  grid_dependency_wait();  // the attention kernel's partial results
  // After a timeout (in that kernel or recorded before it) the partials are incomplete or stale:
  // merge nothing, so that a launch made while the error is recorded leaves the output untouched.
  if (err != nullptr && *reinterpret_cast<const volatile unsigned int*>(err) == kErrTimeout) return;
  const int n_units = static_cast<int>(ws[0]) * kMergeUnitsPerGroup;
  const uint32_t* groups = reinterpret_cast<const uint32_t*>(split_area + split_groups_offset());
  constexpr size_t kSlot = static_cast<size_t>(kBlockM) * (D + 1);
  const float* parts = reinterpret_cast<const float*>(split_area + split_partials_offset());
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int e = static_cast<int>(groups[unit / kMergeUnitsPerGroup]);
    const int t = (unit / (kBlockM / kMergeRows)) & 1;
    const int r0 = (unit % (kBlockM / kMergeRows)) * kMergeRows;
    const SplitEntry en = reinterpret_cast<const SplitEntry*>(split_area)[e];
    const int nch = en.split & 0xffff;
    const int seg_end = en.seg_start + en.seg_len;
    const int row0 = en.q0 + t * kBlockM + r0;
    if (row0 >= seg_end) continue;  // no rows of the item here (uniform across the CTA)
    auto slot = [&](int ch) { return parts + (static_cast<size_t>(e + ch) * 2 + t) * kSlot; };
    __syncthreads();  // the previous unit's weights have been used
    if (threadIdx.x < kMergeRows) {
      const int r = threadIdx.x;
      float l[kSplitMaxChunks];
      float mx = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < kSplitMaxChunks; ++ch) {
        l[ch] = ch < nch ? slot(ch)[static_cast<size_t>(kBlockM) * D + r0 + r] : -INFINITY;
        mx = fmaxf(mx, l[ch]);
      }
      float den = 0.f;
#pragma unroll
      for (int ch = 0; ch < kSplitMaxChunks; ++ch)
        if (ch < nch) den += __expf(l[ch] - mx);
      const float lf = mx + logf(den);
      s_lse[r] = lf;
#pragma unroll
      for (int ch = 0; ch < kSplitMaxChunks; ++ch) s_w[r][ch] = ch < nch ? __expf(l[ch] - lf) : 0.f;
    }
    __syncthreads();
    constexpr int kGroups = D / 8;  // 8 columns (16 bytes of output) per thread and step
    for (int u = threadIdx.x; u < kMergeRows * kGroups; u += kMergeThreads) {
      const int r = u / kGroups, cg = u % kGroups;
      const int q_row = row0 + r;
      if (q_row >= seg_end) continue;
      float4 x[kSplitMaxChunks][2];
#pragma unroll
      for (int ch = 0; ch < kSplitMaxChunks; ++ch) {
        if (ch < nch) {
          const float4* src =
              reinterpret_cast<const float4*>(slot(ch) + static_cast<size_t>(r0 + r) * D + cg * 8);
          x[ch][0] = src[0];
          x[ch][1] = src[1];
        } else {
          x[ch][0] = x[ch][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < kSplitMaxChunks; ++ch) {
        const float w = s_w[r][ch];
        acc[0] = fmaf(w, x[ch][0].x, acc[0]);
        acc[1] = fmaf(w, x[ch][0].y, acc[1]);
        acc[2] = fmaf(w, x[ch][0].z, acc[2]);
        acc[3] = fmaf(w, x[ch][0].w, acc[3]);
        acc[4] = fmaf(w, x[ch][1].x, acc[4]);
        acc[5] = fmaf(w, x[ch][1].y, acc[5]);
        acc[6] = fmaf(w, x[ch][1].z, acc[6]);
        acc[7] = fmaf(w, x[ch][1].w, acc[7]);
      }
      *reinterpret_cast<uint4*>(out + (static_cast<size_t>(q_row) * num_heads + en.head) * D + cg * 8) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                     pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      if (lse != nullptr && cg == 0) lse[static_cast<size_t>(en.head) * capacity + q_row] = s_lse[r];
    }
  }
}

// Exclusive prefix sum over the block (kPlanThreads threads) of one value per thread, and the
// total: a shuffle scan inside each warp, then the warps' totals through shared memory.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* s_warp,
                                                         uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();  // s_warp may still be read from a previous call
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warps' totals (32 warps), total in the last slot
    const uint32_t t = s_warp[lane];
    uint32_t y = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_warp[lane] = y - t;
    if (lane == 31) s_warp[32] = y;
  }
  __syncthreads();
  total = s_warp[32];
  return s_warp[warp] + x - v;
}

__global__ void __launch_bounds__(kPlanThreads)
attn_plan_kernel(const int32_t* __restrict__ cu, int num_segments, int capacity, int max_seqlen,
                 int num_heads, uint32_t* __restrict__ ws, uint8_t* __restrict__ split_area,
                 int wave, unsigned int* err) {
  __shared__ int s_len[kSortMax];
  __shared__ uint32_t s_prefix[kSortMax + 1];   // the item prefix again, for the split's lookups
  __shared__ uint32_t s_warp[kPlanThreads / 32 + 1];
  __shared__ uint32_t s_ngroups;
  grid_dependency_wait();  // cu_seqlens may come from the kernel before this one
  launch_dependents();     // the attention kernel may be scheduled now; it waits for this plan
  const int S = num_segments;
  const int tid = threadIdx.x;
  uint32_t* order = ws + kWsHeader;
  uint32_t* prefix = ws + kWsHeader + S;
  const bool sorted = S <= kSortMax;

  if (sorted) {
    // longest first, ties by position (a stable order): rank = number of segments before it
    for (int g = tid; g < S; g += kPlanThreads)
      s_len[g] = checked_len(cu, g, capacity, max_seqlen, err);
    __syncthreads();
    for (int g = tid; g < S; g += kPlanThreads) {
      int rank = 0;
      for (int h = 0; h < S; ++h) rank += (s_len[h] > s_len[g]) || (s_len[h] == s_len[g] && h < g);
      order[rank] = static_cast<uint32_t>(g);
    }
  } else {
    for (int g = tid; g < S; g += kPlanThreads) order[g] = static_cast<uint32_t>(g);
  }
  __syncthreads();
  auto len_of = [&](int g) {
    return sorted ? s_len[g] : checked_len(cu, g, capacity, max_seqlen, err);
  };

  // exclusive prefix of items over the ordered segments: per-thread chunks + block scan
  const int chunk = (S + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(S, tid * chunk), hi = min(S, lo + chunk);
  uint32_t local = 0;
  for (int i = lo; i < hi; ++i) local += items_of(len_of(static_cast<int>(order[i])), num_heads);
  uint32_t total;
  uint32_t run = block_exclusive_scan(local, s_warp, total);
  for (int i = lo; i < hi; ++i) {
    prefix[i] = run;
    if (sorted) s_prefix[i] = run;
    run += items_of(len_of(static_cast<int>(order[i])), num_heads);
  }
  if (tid == kPlanThreads - 1) {
    prefix[S] = total;
    if (sorted) s_prefix[S] = total;
  }

  // ---- the last wave: items [tail, total) -------------------------------------------------
  const uint32_t tail = wave > 0 ? total / static_cast<uint32_t>(wave) * static_cast<uint32_t>(wave)
                                 : total;
  const uint32_t R = total - tail;
  if (split_area == nullptr || !sorted || R == 0 || R > static_cast<uint32_t>(kSplitMaxEntries) ||
      R > static_cast<uint32_t>(kPlanThreads)) {
    if (tid == 0) {
      ws[0] = 0;
      ws[1] = total;
      ws[2] = total;
      ws[3] = 0;
    }
    return;
  }
  __syncthreads();  // prefix complete
  // thread i < R: whole item tail + i
  int g = 0, a = 0, len = 0, head = 0, q0 = 0, nkv = 0;
  if (tid < static_cast<int>(R)) {
    const uint32_t item = tail + static_cast<uint32_t>(tid);
    int l = 0, h = S - 1;
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (s_prefix[mid] <= item) l = mid; else h = mid - 1;
    }
    g = static_cast<int>(order[l]);
    len = s_len[g];
    a = cu[g];
    const int pairs = (len + kRowsPerItem - 1) / kRowsPerItem;
    const int loc = static_cast<int>(item - s_prefix[l]);
    head = loc / pairs;
    q0 = a + (loc % pairs) * kRowsPerItem;
    nkv = (len + kBlockN - 1) / kBlockN;
  }
  // How many chunks: the L long items of the wave (at least kSplitMinTiles key tiles) are each cut
  // into c = wave / L chunks (at most kSplitMaxChunks, each of at least 4 key tiles), so that
  // their chunks about fill one round of the wave's CTAs; the short items follow them round-robin.
  const bool splittable = tid < static_cast<int>(R) && nkv >= kSplitMinTiles;
  uint32_t n_long;
  block_exclusive_scan(splittable ? 1u : 0u, s_warp, n_long);
  const int c_all = n_long > 0 ? min(kSplitMaxChunks, wave / static_cast<int>(n_long)) : 1;
  int c = tid < static_cast<int>(R) ? (splittable ? max(1, min(c_all, nkv / 4)) : 1) : 0;
  uint32_t E;
  uint32_t first = block_exclusive_scan(static_cast<uint32_t>(c), s_warp, E);
  if (E > static_cast<uint32_t>(kSplitMaxEntries)) {  // too many chunks for the area: stay whole
    c = tid < static_cast<int>(R) ? 1 : 0;
    first = static_cast<uint32_t>(tid);
    E = R;
  }
  SplitEntry* entries = reinterpret_cast<SplitEntry*>(split_area);
  if (tid == 0) s_ngroups = 0u;
  __syncthreads();
  if (c > 1) {  // a split item: list its first entry for the merge (list order is immaterial)
    const uint32_t gi = atomicAdd(&s_ngroups, 1u);
    reinterpret_cast<uint32_t*>(split_area + split_groups_offset())[gi] = first;
  }
  __syncthreads();
  for (int ch = 0; ch < c; ++ch) {
    SplitEntry e;
    e.seg_start = a;
    e.seg_len = len;
    e.head = head;
    e.q0 = q0;
    e.kv0 = nkv * ch / c;
    e.kv1 = nkv * (ch + 1) / c;
    e.group = static_cast<int>(first);
    e.split = c > 1 ? (ch << 16 | c) : 0;
    entries[first + ch] = e;
  }
  if (tid == 0) {
    ws[0] = s_ngroups;
    ws[1] = tail + E;
    ws[2] = tail;
    ws[3] = E;
  }
}

// Item index -> work descriptor: a whole item (binary search of the ordered prefix) or an entry
// of the split last wave.
__device__ __forceinline__ WorkDesc decode_item(uint32_t item, const uint32_t* __restrict__ ws,
                                                const int32_t* __restrict__ cu, int S,
                                                const uint8_t* __restrict__ split_area) {
  WorkDesc d;
  const uint32_t tail = ws[2];
  if (item >= tail) {
    const SplitEntry e = reinterpret_cast<const SplitEntry*>(split_area)[item - tail];
    d.seg_start = e.seg_start;
    d.seg_len = e.seg_len;
    d.head = e.head;
    d.q0 = e.q0;
    d.pk.kv0 = e.kv0;
    d.nkv = e.kv1 - e.kv0;
    d.pk.split = e.split;
    d.pk.group = e.group;
    return d;
  }
  const uint32_t* order = ws + kWsHeader;
  const uint32_t* prefix = ws + kWsHeader + S;
  int lo = 0, hi = S - 1;  // last i with prefix[i] <= item (empty segments repeat a value)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int g = static_cast<int>(order[lo]);
  const int a = cu[g], len = cu[g + 1] - a;
  const uint32_t pairs = static_cast<uint32_t>((len + kRowsPerItem - 1) / kRowsPerItem);
  const uint32_t local = item - prefix[lo];
  d.seg_start = a;
  d.seg_len = len;
  d.head = static_cast<int>(local / pairs);
  d.q0 = a + static_cast<int>(local % pairs) * kRowsPerItem;
  d.pk.kv0 = 0;
  d.nkv = (len + kBlockN - 1) / kBlockN;
  d.pk.split = 0;
  d.pk.group = 0;
  return d;
}

template <int D, int kMode>
struct Cfg {
  static constexpr int kBoxes = D / 64;               // 64-column (128-byte) swizzle boxes
  static constexpr int kTileBytes = kBlockM * D * 2;  // one Q, K or V tile
  static constexpr int kBoxBytes = kBlockM * 128;     // one 128-row box
  // Ring depths (5 tiles of 32 KB fit beside the two Q tiles at D = 128).  Packed segments and
  // VSA: 3 K + 2 V.  Windows: 2 K + 3 V (1-1.5 % faster there).  VSA takes a K and a V tile per
  // query tile per step, so with one producer thread V gained most from depth (50 -> 39 ms on the
  // 1344x768 latent); with V on its own producer thread, K does (34.9 -> 33.9 ms).
  static constexpr int kStagesK = (D == 128) ? (kMode != kModeWindow ? 3 : 2) : 4;
  static constexpr int kStagesV = (D == 128) ? (kMode != kModeWindow ? 2 : 3) : 4;
  // q_full[2], q_empty, k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], s_full[2],
  // p_full[2], o_final[2], o_empty[2], w_full[2], w_empty[2], drain, p_half[2]
  static constexpr int kNumBars = 3 + 2 * kStagesK + 2 * kStagesV + 12 + 1 + 2;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ +
                                    kTileBytes * (kTilesPerItem + kStagesK + kStagesV) +
                                    kNumBars * 8 + 16 /*TMEM slot*/ + 2 * sizeof(WorkDesc);
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(kBlockM, kBlockN, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, true);
};

// VSA: the query blocks of an item's tiles, qb[t][half] (a block past the last repeats the
// tile's first block: its rows are computed and never stored).
__device__ __forceinline__ void vsa_item_blocks(const WorkDesc& d, const WindowAttnGeom& g,
                                                int (&qb)[2][2]) {
  const int last = vsa_num_blocks(g) - 1;
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int h = 0; h < 2; ++h) qb[t][h] = min(d.q0 + 2 * t + h, last);
}

// VSA: one 128-row tile from two blocks' 64-row boxes (block b0 in rows 0-63, b1 in rows 64-127
// of every 64-column half; the 128-byte swizzle repeats every 8 rows, so the halves stack).
template <int kBoxes, int kBoxBytes>
__device__ __forceinline__ void vsa_load_tile(uint8_t* dst, const CUtensorMap* map, int head,
                                              int b0, int b1, uint32_t bar,
                                              const WindowAttnGeom& g) {
  int t0, h0, w0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    vsa_block_origin(half ? b1 : b0, g, t0, h0, w0);
#pragma unroll
    for (int b = 0; b < kBoxes; ++b)
      tma_load_5d(smem_u32(dst + b * kBoxBytes + half * (kBoxBytes / 2)), map, b * 64, head, w0,
                  h0, t0, bar);
  }
}

// kModePacked: packed varlen segments (cu_seqlens, 3-D tensor maps, rows of [capacity, H, D]).
// kModeWindow: windows of a (T, H, W) grid read in place (5-D tensor maps over [T, H, W, heads, D]
// in row-major token order); the output goes back to the same positions.
// kModeVsa: 64-token blocks of the grid read in place; each 64-row half of a query tile is one
// query block.  Key/value tiles follow the pair's schedule (vsa_steps): each step stacks two key
// blocks, and each query block attends to the halves the step marks as its own.  The two query
// tiles of an item have separate key/value streams.
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v,
                const __grid_constant__ CUtensorMap tmap_q2,  // windows: half-height boxes
                const __grid_constant__ CUtensorMap tmap_k2,
                const __grid_constant__ CUtensorMap tmap_v2, __nv_bfloat16* __restrict__ out,
                float* __restrict__ lse, const int32_t* __restrict__ cu_seqlens, int num_segments,
                int capacity, int num_heads, float scale, float scale_log2,
                uint32_t* __restrict__ ws, const __grid_constant__ WindowAttnGeom wg,
                const uint2* __restrict__ vsa_steps, const int2* __restrict__ vsa_counts,
                unsigned int* err, unsigned long long wait_ns, unsigned int stall_after,
                const uint8_t* __restrict__ split_area) {
  constexpr bool kWin = kMode == kModeWindow;
  constexpr bool kVsa = kMode == kModeVsa;
  using C = Cfg<D, kMode>;
  constexpr int SK = C::kStagesK;
  constexpr int SV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                  // 2 tiles
  uint8_t* sK = sQ + kTilesPerItem * C::kTileBytes;    // SK tiles
  uint8_t* sV = sK + SK * C::kTileBytes;               // SV tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + SV * C::kTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  WorkDesc* work = reinterpret_cast<WorkDesc*>(tmem_slot + 4);  // 2-slot ring

  constexpr int kB = 3 + 2 * SK + 2 * SV;  // first per-tile barrier after the rings
  auto bar_qfull = [&](int t) { return smem_u32(&bars[t]); };
  const uint32_t bar_qempty = smem_u32(&bars[2]);
  auto bar_kfull = [&](int s) { return smem_u32(&bars[3 + s]); };
  auto bar_kempty = [&](int s) { return smem_u32(&bars[3 + SK + s]); };
  auto bar_vfull = [&](int s) { return smem_u32(&bars[3 + 2 * SK + s]); };
  auto bar_vempty = [&](int s) { return smem_u32(&bars[3 + 2 * SK + SV + s]); };
  auto bar_sfull = [&](int t) { return smem_u32(&bars[kB + t]); };
  auto bar_pfull = [&](int t) { return smem_u32(&bars[kB + 2 + t]); };
  auto bar_ofinal = [&](int t) { return smem_u32(&bars[kB + 4 + t]); };
  auto bar_oempty = [&](int t) { return smem_u32(&bars[kB + 6 + t]); };
  auto bar_wfull = [&](int i) { return smem_u32(&bars[kB + 8 + i]); };
  auto bar_wempty = [&](int i) { return smem_u32(&bars[kB + 10 + i]); };
  const uint32_t bar_drain = smem_u32(&bars[kB + 12]);
  // P_t over the first 64 keys written (packed and window variants)
  auto bar_phalf = [&](int t) { return smem_u32(&bars[kB + 13 + t]); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Waits of the pipeline give up after wait_ns (2 s unless a test shortens it); the drains at
  // the end always allow the full 2 s, since what they wait for (copies and MMAs already issued)
  // completes by itself.
  auto pwait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, wait_ns); };
  // Testing hook: a producer stops issuing key/value loads once it has issued stall_after tiles
  // (never, by default), as if it had stalled; the waits of the roles that consume them then run
  // out and the kernel unwinds.  Every wait still ends (by its limit) and no access changes.
  bool stalled = false;

  // Everything below reads what earlier kernels wrote (Q/K/V, the plan, the error word).
  grid_dependency_wait();
  launch_dependents();  // the merge kernel may be scheduled; it waits for this kernel to end
  // A wait that timed out earlier (recorded, not yet read) means the machinery is not healthy:
  // leave at once instead of running into 2-second waits again.  The threads decide together, so
  // that a timeout recorded by another CTA meanwhile cannot send some of them on to the set-up
  // barrier without the others.
  if (__syncthreads_or(err != nullptr &&
                       *reinterpret_cast<volatile unsigned int*>(err) == kErrTimeout))
    return;
  // Packed segments: the grid is sized for the most items the capacity allows; a CTA whose first
  // item is past the plan's count has nothing to do, and leaves before any set-up.
  if constexpr (kMode == kModePacked) {
    if (blockIdx.x >= ws[1]) return;
  }

  // ---- setup: barriers (warp 8), TMEM (warp 9) ----
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    if (kWin && wg.half_h) {
      tma_prefetch_desc(&tmap_q2);
      tma_prefetch_desc(&tmap_k2);
      tma_prefetch_desc(&tmap_v2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_qfull(t), 1);
      mbar_init(bar_sfull(t), 1);
      mbar_init(bar_pfull(t), 128);
      mbar_init(bar_phalf(t), 128);
      mbar_init(bar_ofinal(t), 1);
      mbar_init(bar_oempty(t), 128);
      mbar_init(bar_wfull(t), 1);
      // the MMA warp + lane 0 of each of the 8 softmax warps (+ the VSA value producer)
      mbar_init(bar_wempty(t), kVsa ? 10 : 9);
    }
    mbar_init(bar_qempty, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar_kfull(s), 1);
      mbar_init(bar_kempty(s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar_vfull(s), 1);
      mbar_init(bar_vempty(s), 1);
    }
    mbar_init(bar_drain, 1);
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // VSA: stream an item's key (or value) tiles through one ring, per step the tile of query tile
  // 0 then of tile 1 (the order the MMA warp consumes them; a tile whose schedule has ended is
  // skipped); each step's blocks are fetched one step ahead.  K and V have a producer thread each
  // (warps 8 and 10), so a wait on one ring never holds back loads for the other.  Returns false
  // when a wait ran out.
  auto vsa_stream = [&](const WorkDesc& d, auto stages, uint8_t* ring, const CUtensorMap* map,
                        uint32_t full0, uint32_t empty0, uint32_t& cnt) -> bool {
    constexpr int S = decltype(stages)::value;
    const int nt = d.ntiles;
    uint2 cur[2], nxt[2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
      cur[t] = t < nt ? vsa_step(vsa_steps, d.head, d.q0 / 2 + t, 0, wg) : make_uint2(0u, 0u);
    for (int j = 0; j < d.nkv; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t)
        nxt[t] = (t < nt && j + 1 < d.nkv_t[t]) ? vsa_step(vsa_steps, d.head, d.q0 / 2 + t, j + 1, wg)
                                                 : make_uint2(0u, 0u);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t >= nt || j >= d.nkv_t[t]) continue;
        if (cnt >= stall_after) {
          stalled = true;
          return true;
        }
        const uint32_t s = cnt % S;
        if (!pwait(empty0 + 8 * s, ((cnt / S) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(full0 + 8 * s, C::kTileBytes);
        vsa_load_tile<C::kBoxes, C::kBoxBytes>(ring + s * C::kTileBytes, map, d.head,
                                               static_cast<int>(cur[t].x & kVsaBlockMask),
                                               static_cast<int>(cur[t].y & kVsaBlockMask),
                                               full0 + 8 * s, wg);
        ++cnt;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) cur[t] = nxt[t];
    }
    return true;
  };

  if (warp >= 8) {
    setmaxnreg_dec<kRegsOther>();
    if (warp == 8) {
      // ================= scheduler + TMA producer =================
      if (lane == 0) {
        uint32_t total;
        if constexpr (kWin)
          total = static_cast<uint32_t>(wg.nwin[0] * wg.nwin[1] * wg.nwin[2] * num_heads);
        else if constexpr (kVsa)
          total = static_cast<uint32_t>((vsa_num_blocks(wg) + 3) / 4 * num_heads);
        else
          total = ws[1];
        const uint64_t pol_keep = l2_policy_evict_last(), pol_stream = l2_policy_evict_first();
        uint32_t kt = 0, vt = 0;  // K / V tiles loaded so far (positions in the rings)
        uint32_t qn[2] = {0u, 0u};  // Q tiles loaded so far, per tile slot
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const uint32_t item = blockIdx.x + static_cast<uint32_t>(k) * gridDim.x;
          WorkDesc d;
          if (item < total) {
            if constexpr (kWin)
              d = decode_window(item, wg, num_heads);
            else if constexpr (kVsa)
              d = decode_vsa(item, wg, vsa_counts);
            else
              d = decode_item(item, ws, cu_seqlens, num_segments, split_area);
          } else {
            d.seg_start = 0;
            d.seg_len = -1;
            d.head = 0;
            d.q0 = 0;
          }
          ok = pwait(bar_wempty(k & 1), ((k >> 1) & 1) ^ 1);
          if (!ok) break;
          work[k & 1] = d;
          mbar_arrive(bar_wfull(k & 1));
          if (d.seg_len < 0) break;
          const ItemShape sh = shape_of<kMode>(d);
          const bool has1 = sh.has1;
          const int nkv = sh.nkv;
          // tile loads: packed rows [row, row + 128) of one head; window box (w, h, t) of frames,
          // from the half-height map for a half edge window
          const bool hhalf = kWin && d.hbox != wg.w[1];
          // packed segments: every CTA of a (segment, head) streams the same key/value tiles, so
          // they are kept in L2 in preference to the query tiles, which are read once
          auto load_tile = [&](uint8_t* dst, const CUtensorMap* map, int tile, int row,
                               uint32_t bar, uint64_t policy) {
            for (int b = 0; b < C::kBoxes; ++b) {
              if constexpr (kWin)
                tma_load_5d(smem_u32(dst + b * C::kBoxBytes), map, b * 64, d.head, d.box[2],
                            d.box[1], d.box[0] + tile * d.fpt, bar);
              else
                tma_load_3d_hint(smem_u32(dst + b * C::kBoxBytes), map, b * 64, d.head, row, bar,
                                 policy);
            }
          };
          // Q tiles: after the previous item's last QK^T has read the buffers
          ok = pwait(bar_qempty, (k & 1) ^ 1);
          if (!ok) break;
          if constexpr (kVsa) {
            int qb[2][2];
            vsa_item_blocks(d, wg, qb);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t == 1 && !has1) break;
              mbar_arrive_expect_tx(bar_qfull(t), C::kTileBytes);
              vsa_load_tile<C::kBoxes, C::kBoxBytes>(sQ + t * C::kTileBytes, &tmap_q, d.head,
                                                     qb[t][0], qb[t][1], bar_qfull(t), wg);
              ++qn[t];
            }
            ok = vsa_stream(d, std::integral_constant<int, SK>{}, sK, &tmap_k, bar_kfull(0),
                            bar_kempty(0), kt);
            if (stalled) break;
          } else {
            for (int t = 0; t < (has1 ? 2 : 1); ++t) {
              mbar_arrive_expect_tx(bar_qfull(t), C::kTileBytes);
              load_tile(sQ + t * C::kTileBytes, hhalf ? &tmap_q2 : &tmap_q, t, d.q0 + t * kBlockM,
                        bar_qfull(t), pol_stream);
              ++qn[t];
            }
            for (int j = 0; j < nkv && ok; ++j) {
              if (kt >= stall_after) {
                stalled = true;
                break;
              }
              const int row = d.seg_start + (d.pk.kv0 + j) * kBlockN;
              const int s = static_cast<int>(kt % SK);
              ok = pwait(bar_kempty(s), ((kt / SK) & 1) ^ 1);
              if (!ok) break;
              mbar_arrive_expect_tx(bar_kfull(s), C::kTileBytes);
              load_tile(sK + s * C::kTileBytes, hhalf ? &tmap_k2 : &tmap_k, j, row, bar_kfull(s),
                        pol_keep);
              ++kt;
              const int v = static_cast<int>(vt % SV);
              ok = pwait(bar_vempty(v), ((vt / SV) & 1) ^ 1);
              if (!ok) break;
              mbar_arrive_expect_tx(bar_vfull(v), C::kTileBytes);
              load_tile(sV + v * C::kTileBytes, hhalf ? &tmap_v2 : &tmap_v, j, row, bar_vfull(v),
                        pol_keep);
              ++vt;
            }
            if (stalled) break;
          }
        }
        if (!ok) record_error(err, kErrTimeout);
        // Drain: never leave the CTA while a bulk copy may still be landing in shared memory.
        // The last loads of each ring sit on distinct stages, so each stage's latest phase is
        // the one to wait for (already complete in the normal path).
        for (int t = 0; t < 2; ++t)
          if (qn[t] > 0) mbar_wait(bar_qfull(t), (qn[t] - 1) & 1);
        for (uint32_t i = 0; i < SK && i < kt; ++i) {
          const uint32_t x = kt - 1 - i;
          mbar_wait(bar_kfull(x % SK), (x / SK) & 1);
        }
        for (uint32_t i = 0; i < SV && i < vt; ++i) {
          const uint32_t x = vt - 1 - i;
          mbar_wait(bar_vfull(x % SV), (x / SV) & 1);
        }
      }
    } else if (warp == 9) {
      // ================= MMA issuer =================
      // every lane waits and the verdict is made warp-uniform, so the warp never diverges
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, pwait(bar, parity));
      };
      // Two barriers at once: the first polls are issued back to back so their latencies (about
      // 100-200 cycles each, even on a completed phase) overlap instead of adding up.  Used where
      // both are almost always complete when the warp gets there (P and the next K of a packed
      // tile: 41.8 vs 42.4 ms on the H3 request); in the VSA loop polling V, P and K together
      // was 7 % slower and is not done.
      auto wait_all2 = [&](uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1) {
        bool r0 = mbar_try_wait(b0, p0);
        bool r1 = mbar_try_wait(b1, p1);
        if (!r0) r0 = pwait(b0, p0);
        if (!r1) r1 = pwait(b1, p1);
        return __all_sync(0xffffffffu, r0 && r1);
      };

      // Shared-memory descriptors are built once; each MMA adds a compile-time offset (in
      // 16-byte units) to the low half, keeping the single issuing thread's work per MMA small.
      const SmemDesc dq = sw128_desc_split(smem_u32(sQ), 16, 1024);
      const SmemDesc dk = sw128_desc_split(smem_u32(sK), 16, 1024);
      const SmemDesc dv = sw128_desc_split(smem_u32(sV), C::kBoxBytes, 1024);
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      auto issue_qk = [&](int t, int s) {  // S_t = Q_t K_s^T
        const uint32_t d = tmem + kColS + 128 * t;
        const uint32_t qlo = dq.lo + t * kTile16;
        const uint32_t klo = dk.lo + s * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss_split(d, qlo + off, dq.hi, klo + off, dk.hi, C::kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull(t));
      };
      // O_t += P_t V_s over keys [16 kk0, 16 kk1) of the tile
      auto issue_pv = [&](int t, int s, bool first, int kk0 = 0, int kk1 = kBlockN / 16) {
        const uint32_t p = tmem + kColS + 128 * t;
        const uint32_t vlo = dv.lo + s * kTile16;
#pragma unroll
        for (int kk = kk0; kk < kk1; ++kk)
          // 16 keys per MMA: 8 TMEM columns of packed bf16 P; 16 rows (2 KB) of V
          mma_ts_split(tmem + kColO + 128 * t, p + kk * 8, vlo + kk * (2048 >> 4), dv.hi,
                       C::kIdescPV, (!first || kk > 0) ? 1u : 0u);
      };
      const bool leader = elect_one();  // the one thread that issues MMAs and commits

      uint32_t kc = 0, vc = 0;                  // K / V tiles consumed so far
      uint32_t qn[2] = {0u, 0u}, pn[2] = {0u, 0u}, un[2] = {0u, 0u};  // per query tile slot
      bool ok = true, issued = false;
      for (int k = 0; ok; ++k) {
        ok = wait_all(bar_wfull(k & 1), (k >> 1) & 1);
        if (!ok) break;
        const WorkDesc d = work[k & 1];
        __syncwarp();
        if (leader) mbar_arrive(bar_wempty(k & 1));
        if (d.seg_len < 0) break;
        const ItemShape sh = shape_of<kMode>(d);
        const bool has1 = sh.has1;
        const int nkv = sh.nkv;
        const int kv_last_valid = sh.kv_last_valid;  // keys in the last tile (packed)

        if constexpr (kVsa) {
          // Each query tile has its own K/V stream: per step the rings hold K of tile 0, K of
          // tile 1, then V of tile 0, V of tile 1.  Order per step j: PV0_j, S0_{j+1}, PV1_j,
          // S1_{j+1}, as for shared tiles.
          // Tile t runs d.nkv_t[t] steps (its pair's schedule); a tile whose steps have ended is
          // skipped.  The item's last QK^T is step nkv - 1 of the last tile with nkv steps.
          const int nt = has1 ? 2 : 1;
          const int tlast = (has1 && d.nkv_t[1] == nkv) ? 1 : 0;
          ok = wait_all(bar_qfull(0), qn[0]++ & 1);
          if (ok && has1) ok = wait_all(bar_qfull(1), qn[1]++ & 1);
          for (int t = 0; t < nt && ok; ++t) {
            ok = wait_all(bar_kfull(kc % SK), (kc / SK) & 1);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              issue_qk(t, kc % SK);
              mma_commit(bar_kempty(kc % SK));
              if (nkv == 1 && t == nt - 1) mma_commit(bar_qempty);
            }
            issued = true;
            __syncwarp();
            ++kc;
          }
          for (int j = 0; j < nkv && ok; ++j) {
            for (int t = 0; t < nt; ++t) {
              const int nkv_t = t == 0 ? d.nkv_t[0] : d.nkv_t[1];
              if (j >= nkv_t) continue;
              const bool more = j + 1 < nkv_t;
              const int sv = static_cast<int>(vc % SV);
              ok = wait_all(bar_vfull(sv), (vc / SV) & 1);
              if (ok) ok = wait_all(bar_pfull(t), pn[t]++ & 1);
              if (ok && j == 0) ok = wait_all(bar_oempty(t), (un[t] & 1) ^ 1);
              if (ok && more) ok = wait_all(bar_kfull(kc % SK), (kc / SK) & 1);
              if (!ok) break;
              tc_fence_after();
              if (leader) {
                issue_pv(t, sv, j == 0);
                mma_commit(bar_vempty(sv));
                if (!more) mma_commit(bar_ofinal(t));
                if (more) {
                  issue_qk(t, kc % SK);
                  mma_commit(bar_kempty(kc % SK));
                  if (j + 2 == nkv && t == tlast) mma_commit(bar_qempty);
                }
              }
              __syncwarp();
              ++vc;
              if (more) ++kc;
            }
          }
          ++un[0];
          if (has1) ++un[1];
          continue;
        }
        ok = wait_all(bar_qfull(0), qn[0]++ & 1);
        if (ok && has1) ok = wait_all(bar_qfull(1), qn[1]++ & 1);
        if (ok) ok = wait_all(bar_kfull(kc % SK), (kc / SK) & 1);
        if (!ok) break;
        tc_fence_after();
        if (leader) {
          issue_qk(0, kc % SK);
          if (has1) issue_qk(1, kc % SK);
          if (nkv == 1) mma_commit(bar_qempty);  // the item's last QK^T: Q may be reloaded
          mma_commit(bar_kempty(kc % SK));
        }
        issued = true;
        __syncwarp();
        ++kc;
        for (int j = 0; j < nkv && ok; ++j) {
          const int sv = static_cast<int>(vc % SV);
          const bool more = j + 1 < nkv;
          const int sk = static_cast<int>(kc % SK);
          ok = wait_all(bar_vfull(sv), (vc / SV) & 1);
          if (!ok) break;
          if (!kWin && j == nkv - 1 && kv_last_valid < kBlockN) {
            // Zero the value rows past the segment end (rows are 128 B per box; the swizzle only
            // permutes 16-byte chunks within a row, so whole rows are cleared wherever they sit).
            uint8_t* vb = sV + sv * C::kTileBytes;
            const int nrows = kBlockN - kv_last_valid;
            for (int idx = lane; idx < nrows * C::kBoxes * 8; idx += 32) {
              const int r = kv_last_valid + idx / (C::kBoxes * 8);
              const int rem = idx % (C::kBoxes * 8);
              *reinterpret_cast<uint4*>(vb + (rem >> 3) * C::kBoxBytes + r * 128 + (rem & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          // tile 0: PV0_j (the item's first one waits for the previous epilogue), then S0_{j+1}.
          // PV runs in two halves of 64 keys: the first starts as soon as the softmax has
          // written P over those keys, while it still works on the other half.
          ok = wait_all(bar_phalf(0), pn[0] & 1);
          if (ok && j == 0) ok = wait_all(bar_oempty(0), (un[0] & 1) ^ 1);
          if (!ok) break;
          tc_fence_after();
          if (leader) issue_pv(0, sv, j == 0, 0, kBlockN / 32);
          __syncwarp();
          ok = more ? wait_all2(bar_pfull(0), pn[0] & 1, bar_kfull(sk), (kc / SK) & 1)
                    : wait_all(bar_pfull(0), pn[0] & 1);
          ++pn[0];
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            issue_pv(0, sv, j == 0, kBlockN / 32, kBlockN / 16);
            if (!more) mma_commit(bar_ofinal(0));
            if (more) issue_qk(0, sk);
            if (!has1) {
              mma_commit(bar_vempty(sv));
              if (more) mma_commit(bar_kempty(sk));
              if (j + 2 == nkv) mma_commit(bar_qempty);
            }
          }
          __syncwarp();
          if (has1) {
            // tile 1: PV1_j in two halves, then S1_{j+1}
            ok = wait_all(bar_phalf(1), pn[1] & 1);
            if (ok && j == 0) ok = wait_all(bar_oempty(1), (un[1] & 1) ^ 1);
            if (!ok) break;
            tc_fence_after();
            if (leader) issue_pv(1, sv, j == 0, 0, kBlockN / 32);
            __syncwarp();
            ok = wait_all(bar_pfull(1), pn[1]++ & 1);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              issue_pv(1, sv, j == 0, kBlockN / 32, kBlockN / 16);
              mma_commit(bar_vempty(sv));
              if (!more) mma_commit(bar_ofinal(1));
              if (more) {
                issue_qk(1, sk);
                mma_commit(bar_kempty(sk));
                if (j + 2 == nkv) mma_commit(bar_qempty);
              }
            }
            __syncwarp();
          }
          ++vc;
          if (more) ++kc;
        }
        ++un[0];
        if (has1) ++un[1];
      }
      if (!ok && leader) record_error(err, kErrTimeout);
      // Drain: the commit arrives once every MMA issued above has completed, so TMEM is idle
      // before it is released (the normal path has already waited for the last PV).
      if (issued && leader) {
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0);
      }
      __syncwarp();
    } else if (kVsa && warp == 10) {
      // ================= VSA value producer =================
      if (lane == 0) {
        uint32_t vt = 0;  // V tiles loaded so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
          ok = pwait(bar_wfull(k & 1), (k >> 1) & 1);
          if (!ok) break;
          const WorkDesc d = work[k & 1];
          mbar_arrive(bar_wempty(k & 1));
          if (d.seg_len < 0) break;
          ok = vsa_stream(d, std::integral_constant<int, SV>{}, sV, &tmap_v, bar_vfull(0),
                          bar_vempty(0), vt);
          if (stalled) break;
        }
        if (!ok) record_error(err, kErrTimeout);
        for (uint32_t i = 0; i < SV && i < vt; ++i) {  // drain, as for the other producer
          const uint32_t x = vt - 1 - i;
          mbar_wait(bar_vfull(x % SV), (x / SV) & 1);
        }
      }
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ============ softmax / correction / epilogue (warps 0-3: tile 0, 4-7: tile 1) ============
    const int t = warp >> 2;
    const int row = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + kColS + 128 * t;
    const uint32_t o_addr = tmem + lane_base + kColO + 128 * t;
    const float2 c2 = make_float2(scale_log2, scale_log2);
    const uint64_t pol_out = l2_policy_evict_first();
    bool vsa_partial = false;  // VSA: some blocks are cropped by the grid edge (keys need masks)
    if constexpr (kVsa)
      vsa_partial = (wg.L[0] % wg.w[0]) != 0 || (wg.L[1] % wg.w[1]) != 0 || (wg.L[2] % wg.w[2]) != 0;
    uint32_t sn = 0, fn = 0;  // S groups and final-O completions seen by this tile slot
    bool ok = true;
    for (int k = 0; ok; ++k) {
      ok = __all_sync(0xffffffffu, pwait(bar_wfull(k & 1), (k >> 1) & 1));
      if (!ok) break;
      const WorkDesc d = work[k & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_wempty(k & 1));
      if (d.seg_len < 0) break;
      const int seg_end = d.seg_start + d.seg_len;
      const ItemShape sh = shape_of<kMode>(d);
      const bool has1 = sh.has1;
      if (t == 1 && !has1) continue;
      const int nkv = sh.nkv;
      const int kv_last_valid = sh.kv_last_valid;
      // window: which keys of each tile (and which of this tile's query rows) are in the grid
      uint32_t wm0[4], wm1[4];
      if constexpr (kWin) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          wm0[i] = d.mask[0][i];
          wm1[i] = d.mask[1][i];
        }
      }
      float m_used = -INFINITY;  // reference max (raw score units) used in the exponent
      float l = 0.f;
      // New row max mx of step j: move the reference max (and rescale l and O_t) only when it
      // grows by more than 2^kRescaleLog2.  O_t is stable when this runs: PV_t,{j-1} was issued
      // before S_t,j, whose completion the caller observed.
      auto update_max = [&](float mx, int j) {
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * scale_log2 > kRescaleLog2)) {
          alpha = ex2_approx((m_used - mx) * scale_log2);  // 0 when m_used == -inf
          rescale = (j > 0);
          l *= alpha;
          m_used = mx;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t orr[32];
            tmem_ld32(o_addr + c0, orr);
            tmem_ld_wait();
            tmem_reg_fence<32>(orr);
#pragma unroll
            for (int c = 0; c < 32; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
            tmem_st32(o_addr + c0, orr);
          }
        }
      };
      // VSA: this thread's half of the tile (warps 0-1 of the warpgroup: rows 0-63) is query
      // block vqb.  Each step stacks two key blocks (columns 0-63 and 64-127 of S); the step says
      // which of them this query block attends to (one or both), and only those are read.
      const int vhalf = (warp >> 1) & 1;
      int vqb = 0;
      if constexpr (kVsa) vqb = min(d.q0 + 2 * t + vhalf, vsa_num_blocks(wg) - 1);
      const int nsteps = kVsa ? (t == 0 ? d.nkv_t[0] : d.nkv_t[1]) : nkv;
      const int nshared = kVsa ? (t == 0 ? d.nsh_t[0] : d.nsh_t[1]) : 0;
      for (int j = 0; j < nsteps; ++j) {
        uint32_t use0 = 1u, use1 = 1u;          // VSA: this query block's halves of the key tile
        uint64_t vkm0 = ~0ull, vkm1 = ~0ull;    // VSA: their key rows inside the grid
        if constexpr (kVsa) {
          // the schedule's layout: nshared / 2 steps of two shared blocks, the odd shared block
          // in half 0, then this query block's own blocks in its own half
          if (j >= nshared / 2) {
            const bool odd = (nshared & 1) && j == nshared / 2;
            use0 = odd || vhalf == 0;
            use1 = !odd && vhalf == 1;
          }
          if (vsa_partial) {
            const uint2 e = vsa_step(vsa_steps, d.head, d.q0 / 2 + t, j, wg);
            vkm0 = vsa_block_mask(static_cast<int>(e.x & kVsaBlockMask), wg);
            vkm1 = vsa_block_mask(static_cast<int>(e.y & kVsaBlockMask), wg);
          }
        }
        ok = pwait(bar_sfull(t), sn++ & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if constexpr (kVsa) {
          if (!(use0 && use1)) {
            // one key block of the step is this query block's: 64 columns of S
            const int sl = use0 ? 0 : 1;
            const uint64_t vkm = sl ? vkm1 : vkm0;
            uint32_t sr[64];
            tmem_ld32(s_addr + 64 * sl, sr);
            tmem_ld32(s_addr + 64 * sl + 32, sr + 32);
            tmem_ld_wait();
            tmem_reg_fence<64>(sr);
            float s[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c]);
            if (vkm != ~0ull) {
              // key rows of an edge block outside the grid (zero-filled by TMA): -inf by select
#pragma unroll
              for (int c = 0; c < 64; ++c) s[c] = ((vkm >> c) & 1ull) ? s[c] : -INFINITY;
            }
            // row max over the 64 columns: four chains, 3-input steps over 4..59, then 60..63
            float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int c = 4; c < 60; c += 8)
#pragma unroll
              for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[c + u], s[c + 4 + u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], s[60 + u]);
            update_max(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), j);
            const float mb = m_used * scale_log2;
            const float2 nm2 = make_float2(-mb, -mb);
            float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
            uint32_t p[32], z[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, nm2);
              const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              acc[c & 3] = fadd2(acc[c & 3], e);
              p[c] = pack_bf16x2(e.x, e.y);
              z[c] = 0u;
            }
            const float2 a01 = fadd2(acc[0], acc[1]);
            const float2 a23 = fadd2(acc[2], acc[3]);
            l += (a01.x + a01.y) + (a23.x + a23.y);
            // P over S: this block's keys get P, the other block's keys weight 0 for these rows
            tmem_st32(s_addr + 32 * sl, p);
            tmem_st32(s_addr + 32 * (1 - sl), z);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_pfull(t));
            continue;
          }
        }
        uint32_t sr[128];
        tmem_ld32(s_addr + 0, sr + 0);
        tmem_ld32(s_addr + 32, sr + 32);
        tmem_ld32(s_addr + 64, sr + 64);
        tmem_ld32(s_addr + 96, sr + 96);
        tmem_ld_wait();
        tmem_reg_fence<128>(sr);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        if constexpr (kWin) {
          // keys outside the grid (zero-filled rows of an edge window's box): -inf by select
          uint32_t km[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) km[i] = j == 0 ? wm0[i] : wm1[i];
          if ((km[0] & km[1] & km[2] & km[3]) != 0xffffffffu) {
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = ((km[c >> 5] >> (c & 31)) & 1u) ? s[c] : -INFINITY;
          }
        } else if constexpr (kVsa) {
          // key rows of edge blocks outside the grid (zero-filled by TMA): -inf by select
          if ((vkm0 & vkm1) != ~0ull) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              s[c] = (((c < 64 ? vkm0 : vkm1) >> (c & 63)) & 1ull) ? s[c] : -INFINITY;
          }
        } else if (j == nkv - 1 && kv_last_valid < kBlockN) {
          // keys past the segment end: -inf by select, so a NaN/Inf score there is discarded
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c < kv_last_valid) ? s[c] : -INFINITY;
        }
        // row max: four chains, chain u over columns u, u+4, ...: seeded with s[0..3], 3-input
        // steps over columns 4..123, then 124..127
        float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int c = 4; c < 124; c += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], s[c + u], s[c + 4 + u]);
#pragma unroll
        for (int u = 0; u < 4; ++u) m4[u] = fmaxf(m4[u], s[124 + u]);
        update_max(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), j);
        const float mb = m_used * scale_log2;
        const float2 nm2 = make_float2(-mb, -mb);
        float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        uint32_t p[64];
        // P over keys 0-63 first, published on its own so PV can start on it
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, nm2);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[c & 3] = fadd2(acc[c & 3], e);
          p[c] = pack_bf16x2(e.x, e.y);
        }
        if constexpr (!kVsa) {
          tmem_st32(s_addr + 0, p + 0);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar_phalf(t));
        }
#pragma unroll
        for (int c = 32; c < 64; ++c) {
          const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, nm2);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[c & 3] = fadd2(acc[c & 3], e);
          p[c] = pack_bf16x2(e.x, e.y);
        }
        const float2 a01 = fadd2(acc[0], acc[1]);
        const float2 a23 = fadd2(acc[2], acc[3]);
        l += (a01.x + a01.y) + (a23.x + a23.y);
        if constexpr (kVsa) tmem_st32(s_addr + 0, p + 0);  // VSA issues PV in one piece
        tmem_st32(s_addr + 32, p + 32);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pfull(t));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16 rows of this segment; LSE; then O_t is free again ----
      ok = __all_sync(0xffffffffu, pwait(bar_ofinal(t), fn++ & 1));
      if (!ok) break;
      tc_fence_after();
      int q_row;  // this thread's row in the output (original row-major order for windows)
      bool valid;
      if constexpr (kVsa) {
        // row r of the half = (ft * bh + fh) * bw + fw inside query block vqb
        const int r64 = row & (kVsaBlockRows - 1);
        int t0, h0, w0;
        vsa_block_origin(vqb, wg, t0, h0, w0);
        const int gt = t0 + r64 / (wg.w[1] * wg.w[2]);
        const int gh = h0 + (r64 / wg.w[2]) % wg.w[1];
        const int gw = w0 + r64 % wg.w[2];
        valid = d.q0 + 2 * t + vhalf < vsa_num_blocks(wg) && gt < wg.L[0] && gh < wg.L[1] &&
                gw < wg.L[2];
        q_row = (gt * wg.L[1] + gh) * wg.L[2] + gw;
      } else if constexpr (kWin) {
        const int pf = d.hbox * wg.w[2];
        const int gt = d.box[0] + t * d.fpt + row / pf;
        const int gh = d.box[1] + (row / wg.w[2]) % d.hbox;
        const int gw = d.box[2] + row % wg.w[2];
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if ((row >> 5) == i) word = t == 0 ? wm0[i] : wm1[i];
        valid = (word >> (row & 31)) & 1u;
        q_row = (gt * wg.L[1] + gh) * wg.L[2] + gw;
      } else {
        q_row = d.q0 + t * kBlockM + row;
        valid = q_row < seg_end;
      }
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow = out + (static_cast<size_t>(q_row) * num_heads + d.head) * D;
      if constexpr (kMode == kModePacked) {
        if (d.pk.split != 0) {
          // a chunk of a split item: its partial result (O normalised by its own row sum, and
          // its LSE) goes to the split area; attn_merge_kernel combines the chunks afterwards
          constexpr size_t kSlot = static_cast<size_t>(kBlockM) * (D + 1);  // floats per tile
          float* mine = reinterpret_cast<float*>(const_cast<uint8_t*>(split_area) + split_partials_offset()) +
                        (static_cast<size_t>(d.pk.group + (d.pk.split >> 16)) * 2 + t) * kSlot;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t orr[32];
            tmem_ld32(o_addr + c0, orr);
            tmem_ld_wait();
            tmem_reg_fence<32>(orr);
            float4* dst = reinterpret_cast<float4*>(mine + static_cast<size_t>(row) * D + c0);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_float4(__uint_as_float(orr[4 * c]) * inv_l, __uint_as_float(orr[4 * c + 1]) * inv_l,
                                   __uint_as_float(orr[4 * c + 2]) * inv_l, __uint_as_float(orr[4 * c + 3]) * inv_l);
          }
          tc_fence_before();
          mbar_arrive(bar_oempty(t));
          mine[static_cast<size_t>(kBlockM) * D + row] = m_used * scale + logf(l);
          continue;
        }
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t orr[32];
        tmem_ld32(o_addr + c0, orr);
        tmem_ld_wait();
        tmem_reg_fence<32>(orr);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack_bf16x2(__uint_as_float(orr[2 * c]) * inv_l,
                              __uint_as_float(orr[2 * c + 1]) * inv_l);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 val = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            if constexpr (kMode == kModePacked)
              st_global_v4_hint(dst + c, val, pol_out);  // written once: not kept over K/V
            else
              dst[c] = val;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_oempty(t));
      if (lse != nullptr && valid)
        lse[static_cast<size_t>(d.head) * capacity + q_row] = m_used * scale + logf(l);
    }
    if (!ok && lane == 0) record_error(err, kErrTimeout);
  }

  // ---- teardown: every MMA has completed (drained above), then release TMEM ----
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Launch with programmatic stream serialization: the kernel may be scheduled while the previous
// kernel in the stream finishes (it calls grid_dependency_wait() before reading that kernel's
// results), which hides the launch latency between the plan, attention and merge kernels.
template <typename... Params, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int num_sms_of_current_device() {
  static std::atomic<int> cached[64];  // 0 until looked up; racing lookups store the same value
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int D, int kMode>
cudaError_t launch(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<D, kMode>;
  // the shared-memory opt-in is made once per device (a second call from a racing thread is
  // harmless; the flags are atomic so the race is defined)
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, kMode>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return cudaErrorInvalidDevice;
  uint32_t* ws = static_cast<uint32_t*>(a.workspace);
  long long max_items, want;
  if (kMode == kModeWindow) {
    // windows hold at most 256 rows: one CTA per SM looping over (window, head) items
    max_items = static_cast<long long>(a.wg.nwin[0]) * a.wg.nwin[1] * a.wg.nwin[2] * a.num_heads;
    want = sms;
  } else if (kMode == kModeVsa) {
    // four query blocks per item: one CTA per SM looping over (block quad, head) items
    const long long nblk = static_cast<long long>(a.wg.nwin[0]) * a.wg.nwin[1] * a.wg.nwin[2];
    max_items = (nblk + 3) / 4 * a.num_heads;
    want = sms;
  } else {
    e = launch_programmatic(attn_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, a.cu_seqlens,
                            a.num_segments, a.capacity, a.max_seqlen, a.num_heads, ws,
                            static_cast<uint8_t*>(a.split_area), sms, a.err);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // short segments: one CTA per SM (one fits per SM by shared memory and TMEM) looping over
    // items; long segments: one CTA per item.  Never more CTAs than the largest possible number
    // of items (CTAs past the actual count leave at once).
    max_items = (static_cast<long long>(a.capacity) / kRowsPerItem + a.num_segments) * a.num_heads;
    // a job of a few waves at most (whose last wave the plan may split) also loops, so that the
    // short chunks overlap one another's set-up and epilogue
    const bool short_job = max_items <= static_cast<long long>(kPersistMaxWaves) * sms;
    if (a.split_area != nullptr) max_items += kSplitMaxEntries;  // chunks of a split last wave
    want = (a.max_seqlen <= kPersistMaxSeqlen || short_job) ? sms : max_items;
  }
  if (max_items <= 0) return cudaSuccess;
  const int grid = static_cast<int>(max_items < want ? max_items : want);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  const bool half = kMode == kModeWindow && a.wg.half_h;  // the half-height maps were built
  e = launch_programmatic(
      attn_fwd_kernel<D, kMode>, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, a.tmap_q,
      a.tmap_k, a.tmap_v, half ? a.tmap_q2 : a.tmap_q, half ? a.tmap_k2 : a.tmap_k,
      half ? a.tmap_v2 : a.tmap_v, static_cast<__nv_bfloat16*>(a.o), a.lse, a.cu_seqlens,
      a.num_segments, a.capacity, a.num_heads, a.scale, scale_log2, static_cast<uint32_t*>(ws),
      a.wg, a.vsa_steps, a.vsa_counts, a.err, static_cast<unsigned long long>(a.wait_limit_ns),
      a.stall_after_tiles, static_cast<const uint8_t*>(a.split_area));
  if (e != cudaSuccess) return e;
  if (kMode == kModePacked && a.split_area != nullptr)
    e = launch_programmatic(attn_merge_kernel<D>, dim3(4 * sms), dim3(kMergeThreads), 0, stream,
                            static_cast<const uint32_t*>(ws),
                            static_cast<const uint8_t*>(a.split_area),
                            static_cast<__nv_bfloat16*>(a.o), a.lse, a.num_heads, a.capacity,
                            a.err);
  return e;
}

}  // namespace


cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t stream) {
  if (a.mode == kModeWindow) {
    if (a.head_dim == 128) return launch<128, kModeWindow>(a, stream);
    return launch<64, kModeWindow>(a, stream);
  }
  if (a.mode == kModeVsa) {
    if (a.head_dim == 128) return launch<128, kModeVsa>(a, stream);
    return launch<64, kModeVsa>(a, stream);
  }
  if (a.max_seqlen <= 0 || a.num_segments <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch<128, kModePacked>(a, stream);
  return launch<64, kModePacked>(a, stream);
}

}  // namespace h3
