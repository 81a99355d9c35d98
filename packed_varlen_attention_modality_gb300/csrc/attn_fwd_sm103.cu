// Packed varlen (block-diagonal) softmax attention forward for sm_103a: TMA + tcgen05 + TMEM.
//
// [H3-vLLM] "Joint audio/video generation in production: MiniMax-H3 and vLLM-Omni", sec. 3:
// cu_seqlens holds the offsets of the sub-sequences packed into one sequence; a query of
// sub-sequence g softmax-normalises over the keys of g only (no causal mask: the worked
// example's token 15 sees keys 10..29).  Sec. 6: rows past the valid length never take part.
//
// Work unit: one CTA = two 128-row query tiles (256 rows) of one segment and one head; both
// tiles stream the same key/value tiles, so each K/V tile staged in shared memory feeds twice
// the tensor-core work.  No tile crosses a segment boundary: query and key/value tiles start at
// the segment's first row (TMA boxes may start at any row), so only the segment's LAST key tile
// can overhang.  On that tile the overhanging key columns are masked to -inf by select, and
// the overhanging value rows are zeroed in shared memory before the PV product (0 * NaN would
// otherwise leak a neighbour's or a pad row's NaN).  Overhanging query rows are never stored.
//
// Warp roles (384 threads = 3 warpgroups; registers moved to the softmax warpgroups with
// setmaxnreg: 216 each for warpgroups 0 and 1, 72 for warpgroup 2):
//   warps 0-3 / 4-7  softmax of query tile 0 / 1: thread r owns query row r = TMEM lane r and
//              reads its full row of S = Q K^T (128 fp32) with tcgen05.ld, so the row max and
//              row sum need no shuffles.  Running max and sum stay in fp32; P is written back to
//              TMEM over S as bf16 (the A operand of the PV product); O is rescaled in TMEM only
//              when the running max grows by more than 2^8; the epilogue normalises O and
//              stores it (and the LSE).
//   warp 8     TMA producer: Q tiles once, then K and V tiles through rings (3 K / 2 V stages
//              at D = 128).
//   warps 10-11 idle (they complete warpgroup 2).
//   warp 9     MMA issuer (one thread).  Order per key tile j:
//                PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
//              so while softmax 0 works on S0_{j+1} the tensor core runs PV1_j and S1_{j+1},
//              and vice versa (ping-pong).  Because S_t,{j+1} is issued after PV_t,j, seeing
//              S_t,{j+1} complete also means O_t is stable for an in-place rescale.
// TMEM (512 columns): O0 [0,128), O1 [128,256), S0/P0 [256,384), S1/P1 [384,512).
#include <cuda_bf16.h>

#include "h3_internal.h"
#include "sm103_ptx.cuh"

namespace h3 {
namespace {

constexpr int kBlockM = 128;          // query rows per tile
constexpr int kBlockN = 128;          // keys per tile
constexpr int kTilesPerCta = 2;       // query tiles per CTA
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 216;  // 128 * (216 + 216 + 72) = 384 * 168 registers at launch
constexpr int kRegsOther = 72;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;              // O of tile t at kColO + 128 t
constexpr int kColS = 256;            // S / P of tile t at kColS + 128 t
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the running max grows by > 2^8

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;               // 64-column (128-byte) swizzle boxes
  static constexpr int kTileBytes = kBlockM * D * 2;  // one Q, K or V tile
  static constexpr int kBoxBytes = kBlockM * 128;     // one 128-row box
  static constexpr int kStagesK = (D == 128) ? 3 : 4;  // K ring depth
  static constexpr int kStagesV = (D == 128) ? 2 : 4;  // V ring depth
  // q_full[2], k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], s_full[2], p_full[2],
  // o_final[2], drain
  static constexpr int kNumBars = 2 + 2 * kStagesK + 2 * kStagesV + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ +
                                    kTileBytes * (kTilesPerCta + kStagesK + kStagesV) +
                                    kNumBars * 8 + 16;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(kBlockM, kBlockN, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, true);
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, __nv_bfloat16* __restrict__ out,
                float* __restrict__ lse, const int32_t* __restrict__ cu_seqlens, int capacity,
                int num_heads, float scale, float scale_log2, unsigned int* err) {
  using C = Cfg<D>;
  constexpr int SK = C::kStagesK;
  constexpr int SV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                  // 2 tiles
  uint8_t* sK = sQ + kTilesPerCta * C::kTileBytes;     // SK tiles
  uint8_t* sV = sK + SK * C::kTileBytes;               // SV tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + SV * C::kTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);

  auto bar_qfull = [&](int t) { return smem_u32(&bars[t]); };
  constexpr int kB = 2 + 2 * SK + 2 * SV;  // first per-tile barrier after the rings
  auto bar_kfull = [&](int s) { return smem_u32(&bars[2 + s]); };
  auto bar_kempty = [&](int s) { return smem_u32(&bars[2 + SK + s]); };
  auto bar_vfull = [&](int s) { return smem_u32(&bars[2 + 2 * SK + s]); };
  auto bar_vempty = [&](int s) { return smem_u32(&bars[2 + 2 * SK + SV + s]); };
  auto bar_sfull = [&](int t) { return smem_u32(&bars[kB + t]); };
  auto bar_pfull = [&](int t) { return smem_u32(&bars[kB + 2 + t]); };
  auto bar_ofinal = [&](int t) { return smem_u32(&bars[kB + 4 + t]); };
  const uint32_t bar_drain = smem_u32(&bars[kB + 6]);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x;  // query tiles 2*pair and 2*pair+1 of the segment
  const int head = blockIdx.y;
  const int seg = blockIdx.z;

  // A wait that timed out earlier (recorded, not yet read) means the machinery is not healthy:
  // every later CTA leaves at once instead of running into its own 2-second waits.
  if (err != nullptr && *reinterpret_cast<volatile unsigned int*>(err) == kErrTimeout) return;

  // ---- segment bounds (device-side validation; uniform across the CTA) ----
  const int seg_start = cu_seqlens[seg];
  const int seg_end = cu_seqlens[seg + 1];
  const bool bad = seg_start < 0 || seg_end < seg_start || seg_end > capacity ||
                   (seg == 0 && seg_start != 0);
  if (bad) {
    if (threadIdx.x == 0 && pair == 0 && head == 0) record_error(err, kErrBadCuSeqlens);
    return;
  }
  const int seg_len = seg_end - seg_start;
  if (pair == static_cast<int>(gridDim.x) - 1 && threadIdx.x == 0 && head == 0 &&
      seg_len > static_cast<int>(gridDim.x) * kTilesPerCta * kBlockM)
    record_error(err, kErrBadCuSeqlens);  // max_seqlen smaller than a segment
  const int q0 = seg_start + pair * kTilesPerCta * kBlockM;
  if (q0 >= seg_end) return;
  const bool has1 = q0 + kBlockM < seg_end;  // second query tile present
  const int nkv = (seg_len + kBlockN - 1) / kBlockN;
  const int kv_last_valid = seg_len - (nkv - 1) * kBlockN;  // keys in the last tile, 1..128

  // ---- setup: barriers (warp 8), TMEM (warp 9) ----
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_qfull(t), 1);
      mbar_init(bar_sfull(t), 1);
      mbar_init(bar_pfull(t), 128);
      mbar_init(bar_ofinal(t), 1);
    }
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

  if (warp >= 8) {
    setmaxnreg_dec<kRegsOther>();
    if (warp == 8) {
      // ================= TMA producer =================
      if (lane == 0) {
        int issued_k = 0, issued_v = 0;
        bool ok = true;
        for (int t = 0; t < (has1 ? 2 : 1); ++t) {
          mbar_arrive_expect_tx(bar_qfull(t), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem_u32(sQ + t * C::kTileBytes + b * C::kBoxBytes), &tmap_q, b * 64, head,
                        q0 + t * kBlockM, bar_qfull(t));
        }
        for (int j = 0; j < nkv; ++j) {
          const int row = seg_start + j * kBlockN;
          const int s = j % SK;
          ok = mbar_wait(bar_kempty(s), ((j / SK) & 1) ^ 1);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_kfull(s), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem_u32(sK + s * C::kTileBytes + b * C::kBoxBytes), &tmap_k, b * 64, head,
                        row, bar_kfull(s));
          issued_k = j + 1;
          const int v = j % SV;
          ok = mbar_wait(bar_vempty(v), ((j / SV) & 1) ^ 1);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_vfull(v), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(smem_u32(sV + v * C::kTileBytes + b * C::kBoxBytes), &tmap_v, b * 64, head,
                        row, bar_vfull(v));
          issued_v = j + 1;
        }
        if (!ok) record_error(err, kErrTimeout);
        // Drain: never leave the CTA while a bulk copy may still be landing in shared memory.
        // The last S loads of each kind sit on distinct stages, so each stage's latest phase is
        // the one to wait for (already complete in the normal path).
        for (int t = 0; t < (has1 ? 2 : 1); ++t) mbar_wait(bar_qfull(t), 0);
        for (int j = issued_k - 1; j >= 0 && j >= issued_k - SK; --j)
          mbar_wait(bar_kfull(j % SK), (j / SK) & 1);
        for (int j = issued_v - 1; j >= 0 && j >= issued_v - SV; --j)
          mbar_wait(bar_vfull(j % SV), (j / SV) & 1);
      }
    } else if (warp == 9) {
      // ================= MMA issuer =================
      // every lane waits and the verdict is made warp-uniform, so the warp never diverges
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity));
      };
      const uint32_t qa0 = smem_u32(sQ);
      auto issue_qk = [&](int t, int s) {  // S_t = Q_t K_s^T
        const uint32_t d = tmem + kColS + 128 * t;
        const uint32_t qa = qa0 + t * C::kTileBytes;
        const uint32_t kb = smem_u32(sK + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
          mma_ss(d, sw128_desc(qa + off, 16, 1024), sw128_desc(kb + off, 16, 1024), C::kIdescQK,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(bar_sfull(t));
      };
      auto issue_pv = [&](int t, int s, bool first) {  // O_t += P_t V_s
        const uint32_t p = tmem + kColS + 128 * t;
        const uint32_t vb = smem_u32(sV + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          // 16 keys per MMA: 8 TMEM columns of packed bf16 P; 16 rows (2 KB) of V
          mma_ts(tmem + kColO + 128 * t, p + kk * 8, sw128_desc(vb + kk * 2048, C::kBoxBytes, 1024),
                 C::kIdescPV, (!first || kk > 0) ? 1u : 0u);
      };

      bool ok = wait_all(bar_qfull(0), 0);
      if (ok && has1) ok = wait_all(bar_qfull(1), 0);
      if (ok) ok = wait_all(bar_kfull(0), 0);
      if (ok) {
        tc_fence_after();
        if (lane == 0) {
          issue_qk(0, 0);
          if (has1) issue_qk(1, 0);
          mma_commit(bar_kempty(0));
        }
        __syncwarp();
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int sv = j % SV;
        const bool more = j + 1 < nkv;
        const int sk = (j + 1) % SK;
        ok = wait_all(bar_vfull(sv), (j / SV) & 1);
        if (!ok) break;
        if (j == nkv - 1 && kv_last_valid < kBlockN) {
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
        // tile 0: PV0_j, then S0_{j+1}
        ok = wait_all(bar_pfull(0), j & 1);
        if (!ok) break;
        if (more) ok = wait_all(bar_kfull(sk), ((j + 1) / SK) & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          issue_pv(0, sv, j == 0);
          if (!more) mma_commit(bar_ofinal(0));
          if (more) issue_qk(0, sk);
          if (!has1) {
            mma_commit(bar_vempty(sv));
            if (more) mma_commit(bar_kempty(sk));
          }
        }
        __syncwarp();
        if (has1) {
          // tile 1: PV1_j, then S1_{j+1}
          ok = wait_all(bar_pfull(1), j & 1);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            issue_pv(1, sv, j == 0);
            mma_commit(bar_vempty(sv));
            if (!more) mma_commit(bar_ofinal(1));
            if (more) {
              issue_qk(1, sk);
              mma_commit(bar_kempty(sk));
            }
          }
          __syncwarp();
        }
      }
      if (!ok && lane == 0) record_error(err, kErrTimeout);
      // Drain: the commit arrives once every MMA issued above has completed, so TMEM is idle
      // before it is released (the normal path has already waited for the last PV).
      if (lane == 0) {
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0);
      }
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    if (warp < 4 || has1) {
      // ============ softmax / correction / epilogue (warps 0-3: tile 0, 4-7: tile 1) ============
      const int t = warp >> 2;
      const int row = threadIdx.x & 127;  // query row within the tile == TMEM lane
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t s_addr = tmem + lane_base + kColS + 128 * t;
      const uint32_t o_addr = tmem + lane_base + kColO + 128 * t;
      const float2 c2 = make_float2(scale_log2, scale_log2);
      float m_used = -INFINITY;  // reference max (raw score units) used in the exponent
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        ok = mbar_wait(bar_sfull(t), j & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
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
        if (j == nkv - 1 && kv_last_valid < kBlockN) {
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
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * scale_log2 > kRescaleLog2)) {
          alpha = ex2_approx((m_used - mx) * scale_log2);  // 0 when m_used == -inf
          rescale = (j > 0);
          l *= alpha;
          m_used = mx;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O_t is stable: PV_t,{j-1} was issued before S_t,j, whose completion we observed.
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
        const float mb = m_used * scale_log2;
        const float2 nm2 = make_float2(-mb, -mb);
        float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        uint32_t p[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), c2, nm2);
          const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[c & 3] = fadd2(acc[c & 3], e);
          p[c] = pack_bf16x2(e.x, e.y);
        }
        const float2 a01 = fadd2(acc[0], acc[1]);
        const float2 a23 = fadd2(acc[2], acc[3]);
        l += (a01.x + a01.y) + (a23.x + a23.y);
        tmem_st32(s_addr + 0, p + 0);
        tmem_st32(s_addr + 32, p + 32);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_pfull(t));
      }
      // ---- epilogue: O / l -> bf16 rows of this segment; LSE ----
      if (ok) {
        ok = mbar_wait(bar_ofinal(t), 0);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        const int q_row = q0 + t * kBlockM + row;
        const bool valid = q_row < seg_end;
        const float inv_l = 1.f / l;
        __nv_bfloat16* orow = out + (static_cast<size_t>(q_row) * num_heads + head) * D;
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
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          }
        }
        if (lse != nullptr && valid)
          lse[static_cast<size_t>(head) * capacity + q_row] = m_used * scale + logf(l);
      } else if (lane == 0) {
        record_error(err, kErrTimeout);
      }
    }
  }

  // ---- teardown: every MMA has completed (drained above), then release TMEM ----
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool configured[64] = {};  // the shared-memory opt-in is made once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int qtiles = (a.max_seqlen + kBlockM - 1) / kBlockM;
  const dim3 grid((qtiles + kTilesPerCta - 1) / kTilesPerCta, a.num_heads, a.num_segments);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  attn_fwd_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(
      a.tmap_q, a.tmap_k, a.tmap_v, static_cast<__nv_bfloat16*>(a.o), a.lse, a.cu_seqlens,
      a.capacity, a.num_heads, a.scale, scale_log2, a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& a, cudaStream_t stream) {
  if (a.max_seqlen <= 0 || a.num_segments <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch<128>(a, stream);
  return launch<64>(a, stream);
}

}  // namespace h3
