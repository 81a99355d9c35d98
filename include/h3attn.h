/*
 * h3attn -- packed varlen attention with modality-tagged 3D RoPE, for GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Every buffer is owned by the caller; the library
 * allocates no device memory except one 4-byte error word per device (a static __device__
 * variable), and keeps no state between calls except cached driver entry points.
 *
 * Sources (page title + section):
 *   [H3-vLLM] "Joint audio/video generation in production: MiniMax-H3 and vLLM-Omni"
 *       sec. 3 "Packed sequence and modality identity": one packed 1-D sequence of text,
 *       audio and video rows; cu_seqlens holds the sub-sequence offsets; the kernel makes each
 *       sub-sequence softmax over its own keys only (worked example [0,10,30] -> [0,10,30,45]);
 *       a per-token modality tag selects the RoPE treatment.
 *       sec. 6 "Boundary trim of packed attention": only the valid length (58,758 of an aligned
 *       58,816) may enter the kernel; the trim changes a length and a pointer, copies nothing.
 *   [H3-fast] "Breaking the engineering bottlenecks of video-generation models"
 *       "Crossing the time boundary", step 3: t_global = t_local + s * 40/24 before RoPE,
 *       time axis only, decimals kept.
 *       "Breaking the memory wall: window attention across GPUs": regular and half-shifted
 *       3D windows with cropped edge windows; tokens gathered per window, order restored.
 *
 * Conventions for every call:
 *   - Tensors Q, K, V, O are bf16, row-major [C, H, D]: token stride H*D elements, D contiguous.
 *     C (capacity) >= N (valid tokens) -- rows in [N, C) are padding: never read as keys or
 *     values that contribute, never written.
 *   - Device pointers must be 16-byte aligned; head_dim must be 64 or 128.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).  They
 *     return after host-side validation of scalars and pointers.  A status other than H3_OK
 *     means nothing was launched.
 *   - Device-side contents (cu_seqlens, perm) are checked by the kernels: a bad value makes
 *     the kernel skip the affected work and record an error code in the device error word,
 *     never access memory out of bounds.  h3_get_device_error() reads (and clears) that word.
 *   - No exceptions cross the ABI; nothing aborts; no device trap.
 *   - The library looks up the device addresses of its own device variables (the error word,
 *     the array of h3_varlen_attn_fwd_noalloc) once per device and keeps them for the life of
 *     the process.  Do not use it across a cudaDeviceReset (or any other destruction of a
 *     device's primary context): the variables would then live at new addresses.
 */
#ifndef H3ATTN_H_
#define H3ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define H3_API __attribute__((visibility("default")))
#else
#define H3_API
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* h3_stream_t;

typedef enum {
  H3_OK = 0,
  H3_ERR_NULL = 1,            /* a required pointer is NULL */
  H3_ERR_INVALID_ARG = 2,     /* a size or scalar is out of range */
  H3_ERR_BAD_CU_SEQLENS = 3,  /* (device) cu_seqlens not 0-based, decreasing, beyond capacity,
                                 or a segment longer than max_seqlen */
  H3_ERR_UNSUPPORTED = 4,     /* head_dim not in {64, 128}, or no sm_103a device */
  H3_ERR_WORKSPACE = 5,       /* workspace missing or too small */
  H3_ERR_CUDA = 6,            /* a CUDA runtime / driver call failed */
  H3_ERR_TIMEOUT = 7,         /* (device) a bounded wait inside a kernel ran out */
  H3_ERR_MISALIGNED = 8,      /* a device pointer or row size is not 16-byte aligned */
  H3_ERR_BAD_PERM = 9,        /* (device) a permutation entry is out of range */
  H3_ERR_BAD_BLOCK_INDEX = 10 /* (device) a selected VSA block index is out of range */
} h3_status;

enum { H3_TAG_TEXT = 0, H3_TAG_VIDEO = 1, H3_TAG_AUDIO = 2 };

/* RoPE configuration ([H3-vLLM] sec. 3: the tag selects the frequencies).
 * Zero / negative fields select the defaults given in brackets. */
typedef struct {
  float base_text;      /* [10000] ladder base of text rows: one band over all D dims, by t */
  float base_video;     /* [10000] ladder base of each video band */
  float base_audio;     /* [10000] ladder base of audio rows: one band over all D dims, by t */
  int32_t video_dims_t; /* video band widths, must sum to head_dim and be even;   */
  int32_t video_dims_h; /*   all three 0 selects D/2 : D/4 : D/4                   */
  int32_t video_dims_w; /*   (32/16/16 at D = 64, 64/32/32 at D = 128)           */
  float audio_hz;       /* [40] numerator of the continuation shift ratio  ([H3-fast])   */
  float video_fps;      /* [24] denominator of the continuation shift ratio            */
} h3_rope_cfg;

/* Modality-tagged rotary position encoding of Q and K, with the continuation time shift.
 *
 * [H3-vLLM] sec. 3 (tags choose the RoPE treatment; modality position spaces independent) and
 * [H3-fast] "Crossing the time boundary" step 3 (t_global = t_local + s * 40/24, time only).
 *
 * For token i of request r with tag tau and local position (t, h, w) = pos[i]:
 *   t_g = t + s_r * audio_hz / video_fps   (s_r = start_frames[r]; fp32, correctly rounded)
 *   pairs (x[2j], x[2j+1]) are rotated by phi_j:
 *     text / audio : phi_j = t_g * base^(-2j/D),                  j in [0, D/2)
 *     video        : band t dims [0,d_t): t_g * base^(-2j/d_t); band h: h * base^(-2j/d_h);
 *                    band w: w * base^(-2j/d_w)   (j counts pairs within the band)
 *   x'[2j] = x[2j] cos phi - x[2j+1] sin phi;   x'[2j+1] = x[2j] sin phi + x[2j+1] cos phi
 *
 * q_in, q_out : device bf16 [C, H, D]; q_out may equal q_in (in place) but must not otherwise
 *               overlap it.  Only rows [0, num_tokens) are read and written.
 * k_in, k_out : same for K; both NULL to rotate Q only.
 * pos         : device fp32 [num_tokens, 3] local (t, h, w); h, w ignored for text/audio.
 * tag         : device uint8 [num_tokens]; values other than 1 (video) / 2 (audio) act as text.
 * cu_requests : device int32 [num_requests + 1], request row offsets (0-based, non-decreasing,
 *               last = num_tokens); NULL means one request covering every row.
 * start_frames: device fp32 [num_requests], continuation start frame s_r; NULL means all 0.
 * cfg         : host pointer, or NULL for all defaults.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_UNSUPPORTED, H3_ERR_MISALIGNED, H3_ERR_CUDA.
 */
H3_API h3_status h3_rope_apply(const void* q_in, void* q_out, const void* k_in, void* k_out,
                        int32_t num_tokens, int32_t num_heads, int32_t head_dim,
                        const float* pos, const uint8_t* tag,
                        const int32_t* cu_requests, int32_t num_requests,
                        const float* start_frames, const h3_rope_cfg* cfg, h3_stream_t stream);

/* Bytes of device workspace h3_varlen_attn_fwd wants for these sizes: the work plan written by
 * the call itself (segment order and item prefix, 8 bytes per segment, plus a 16-byte header,
 * rounded up to 256) and, when max_seqlen >= 1024, a split area after it (about 42 MB at
 * head_dim 128, 21 MB at 64).  With the split area the call may cut the long work items of its
 * last, partly filled wave of CTAs into chunks of their key range, so that the wave spreads over
 * every SM; the chunks' partial results are merged in a fixed order, so the output does not
 * depend on which chunk finishes last.  The plan alone (the size returned for max_seqlen < 1024)
 * is the minimum the call accepts; it then never splits.  0 when num_segments <= 0. */
H3_API size_t h3_varlen_attn_workspace_size(int32_t num_segments, int32_t num_heads,
                                     int32_t max_seqlen, int32_t head_dim);

/* Block-diagonal (packed varlen) softmax attention forward, non-causal.
 *
 * [H3-vLLM] sec. 3: for segment g = [cu[g], cu[g+1]), head h and query row i in g,
 *   S_ij = scale * <q_i, k_j> for j in g only;  P = softmax_j(S);  o_i = sum_j P_ij v_j;
 *   lse_i = log sum_j exp(S_ij).  Keys outside g get weight exactly zero (they are never
 *   multiplied in, so NaN/Inf there cannot leak).  [H3-vLLM] sec. 6: rows >= cu[S] are never
 *   read as contributing keys/values and never written (trim = length only, no copy).
 *
 * q, k, v     : device bf16 [capacity, H, D].
 * o           : device bf16 [capacity, H, D]; rows of every segment written, others untouched.
 * lse         : device fp32 [H, capacity] (natural log) or NULL.
 * cu_seqlens  : device int32 [num_segments + 1]; must start at 0, not decrease, end <= capacity.
 *               Empty segments are allowed.
 * max_seqlen  : host upper bound on the longest segment.  A longer segment is still computed in
 *               full but reported as H3_ERR_BAD_CU_SEQLENS.
 * softmax_scale: <= 0 selects 1/sqrt(head_dim).
 * workspace   : device scratch of h3_varlen_attn_workspace_size() bytes (16-byte aligned), or
 *               NULL when that size is 0; at least the plan (see there).  Contents need not be
 *               initialised; the call rewrites what it reads.  Calls that may run at the same
 *               time (other streams) need separate workspaces.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_UNSUPPORTED, H3_ERR_MISALIGNED,
 *         H3_ERR_WORKSPACE, H3_ERR_CUDA; device-side H3_ERR_BAD_CU_SEQLENS / H3_ERR_TIMEOUT.
 */
H3_API h3_status h3_varlen_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* cu_seqlens, int32_t num_segments, int32_t max_seqlen,
                             int32_t capacity, int32_t num_heads, int32_t head_dim,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             h3_stream_t stream);

/* Largest num_segments h3_varlen_attn_fwd_noalloc accepts. */
#define H3_NOALLOC_MAX_SEGMENTS 16384

/* h3_varlen_attn_fwd without a workspace argument, for callers that cannot allocate device
 * memory -- for example code running where a cudaMalloc would synchronise the device or is not
 * permitted (inside a caller's own memory pool or allocator, a plugin host that owns all device
 * memory, a latency-critical loop).  The pages have no counterpart: this is a convenience of the
 * library, not a step of the method.
 *
 * Same inputs, outputs, semantics and errors as h3_varlen_attn_fwd.  Instead of a workspace it
 * uses a fixed array inside the library (132 KB per device, held from the first use until the
 * process exits), so it calls no cudaMalloc, cudaFree or other allocating routine.  The array
 * holds the plan alone, so work items are never split: the result is, bit for bit, that of
 * h3_varlen_attn_fwd given a plan-only workspace.
 *   - At most H3_NOALLOC_MAX_SEGMENTS segments; more returns H3_ERR_WORKSPACE, launching nothing.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls on a device share the array.  Calls whose kernels may overlap on the GPU (other
 *     streams, other host threads) race on it and must not be issued; serialise them, or use
 *     h3_varlen_attn_fwd with a workspace per stream.
 *   - Each call rewrites every part of the array it reads, so nothing needs clearing between
 *     calls. */
H3_API h3_status h3_varlen_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                            float* lse, const int32_t* cu_seqlens,
                                            int32_t num_segments, int32_t max_seqlen,
                                            int32_t capacity, int32_t num_heads, int32_t head_dim,
                                            float softmax_scale, h3_stream_t stream);

/* Number of windows of the partition (host only; no device work).
 * [H3-fast] "window attention across GPUs": along each axis of length L with window w and
 * shift s there are ceil((L + s) / w) windows (edge windows cropped).  Returns -1 on bad input
 * (non-positive grid or window, shift < 0 or >= window). */
H3_API int32_t h3_window_count(const int32_t grid[3], const int32_t win[3], const int32_t shift[3]);

/* Shifted 3D window partition + gather of rows into per-window segments.
 *
 * [H3-fast] "window attention across GPUs": the (T, H, W) token grid (row-major order) is cut
 * into windows; token (t, h, w) belongs to axis windows floor((x + s) / w); windows are
 * numbered lexicographically (i_t, i_h, i_w); the packed order lists windows by number and,
 * inside a window, tokens by their original row-major index.
 *
 * grid, win, shift: host int32[3] each (T, H, W order).
 * perm       : device int32 [N] out, perm[j] = original row of packed row j (N = T*H*W).
 * cu_seqlens : device int32 [nwin + 1] out (nwin = h3_window_count()).
 * src, dst   : host arrays of num_tensors device pointers; dst[i] row j = src[i] row perm[j].
 *              Each tensor is [N, row_bytes]; dst must not overlap src.  num_tensors may be 0
 *              (indexing only), at most 8.
 * row_bytes  : bytes per row (e.g. H * D * 2), a positive multiple of 16.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_MISALIGNED, H3_ERR_CUDA.
 */
H3_API h3_status h3_window_pack(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                         int32_t* perm, int32_t* cu_seqlens,
                         const void* const* src, void* const* dst, int32_t num_tensors,
                         int32_t row_bytes, h3_stream_t stream);

/* Shifted 3D window attention computed in place on the grid: the same result as
 * h3_window_pack -> h3_varlen_attn_fwd over the window segments -> h3_window_unpack, without the
 * packed copies.
 *
 * [H3-fast] "window attention across GPUs": every window of the (T, H, W) grid (windows win,
 * shifted by shift, edge windows cropped) attends within itself; the output stays in the
 * original token order.  Each window's rows are read straight from the grid with 5-D tensor
 * loads (a 128-row tile = whole frames of one window); rows of an edge window's box that fall
 * outside the grid are never used as keys and never written.
 *
 * q, k, v, o : device bf16 [T*H*W, num_heads, head_dim], rows in row-major (t, h, w) order.
 * lse        : device fp32 [num_heads, T*H*W] (natural log) or NULL.
 * grid, win, shift : host int32[3] each; as for h3_window_pack.  Supported windows: win[1]*win[2]
 *              divides 128 and win[0]*win[1]*win[2] <= 256 (e.g. 4x8x8); else H3_ERR_UNSUPPORTED.
 * softmax_scale: <= 0 selects 1/sqrt(head_dim).  No workspace.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_UNSUPPORTED, H3_ERR_MISALIGNED, H3_ERR_CUDA.
 */
H3_API h3_status h3_window_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                    const int32_t grid[3], const int32_t win[3],
                                    const int32_t shift[3], int32_t num_heads, int32_t head_dim,
                                    float softmax_scale, h3_stream_t stream);

/* Restore original token order: dst row perm[j] = src row j, for j in [0, num_tokens).
 * [H3-fast] "window attention across GPUs" (token order restored after attention).
 * perm is device int32 [num_tokens] (a permutation of [0, num_tokens); an entry out of range is
 * skipped and recorded as H3_ERR_BAD_PERM).  src, dst device [num_tokens, row_bytes], disjoint.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_MISALIGNED, H3_ERR_CUDA. */
H3_API h3_status h3_window_unpack(const int32_t* perm, int32_t num_tokens, const void* src, void* dst,
                           int32_t row_bytes, h3_stream_t stream);

/* ---- Block-sparse video attention (VSA) ----------------------------------------------------
 * [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section "VSA:
 * block-sparse attention": the video latent is cut into 4x4x4 = 64-token blocks along time,
 * height and width; a block-level gate scores each key block against the query block and only
 * the top-k blocks enter a token-level attention between the selected blocks.  The pages leave
 * the gate and k open: here the gate score of key block b for query block a (per head) is
 * scale * <mean of a's query rows, mean of b's key rows>, means over the block's tokens inside the
 * grid; k is the caller's.
 *
 * Layout shared by the VSA calls: q, k, v, o are device bf16 [T*H*W, num_heads, head_dim] in
 * row-major (t, h, w) token order (the layout of h3_window_attn_fwd).  Blocks are cut at
 * multiples of block[] from the origin (no shift), edge blocks cropped by the grid; block id
 * = (i_t * nb_h + i_h) * nb_w + i_w with nb_a = ceil(grid[a] / block[a]).
 * Supported: block[0] * block[1] * block[2] == 64 (e.g. 4x4x4), head_dim 64 or 128; else
 * H3_ERR_UNSUPPORTED. */

/* Number of blocks: prod ceil(grid[a] / block[a]); -1 for a non-positive size or overflow. */
H3_API int32_t h3_vsa_block_count(const int32_t grid[3], const int32_t block[3]);

/* Workspace bytes of h3_vsa_select (the block means of Q and K, fp32); 0 for invalid sizes. */
H3_API size_t h3_vsa_select_workspace_size(const int32_t grid[3], const int32_t block[3],
                                           int32_t num_heads, int32_t head_dim);

/* Block gate scores and top-k block selection.
 * q, k       : device bf16 [T*H*W, num_heads, head_dim] (layout above); 16-byte aligned.
 * topk       : selected key blocks per query block, 1 <= topk <= nblk.
 * softmax_scale: scale of the gate scores; <= 0 selects 1/sqrt(head_dim).
 * scores     : device fp32 [num_heads, nblk, nblk] out, caller-owned: the gate scores.
 * block_idx  : device int32 [num_heads, nblk, topk] out: for each head and query block, the
 *              topk key blocks with the highest scores (equal scores: lower block id first),
 *              listed in ascending block id.
 * workspace  : device, >= h3_vsa_select_workspace_size() bytes, 16-byte aligned.
 * Scores are accumulated in fp32 (block means in token order, dot products in dimension order),
 * so blocks whose scores differ by fp32 rounding may be taken in either order.  Inputs must be
 * finite.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_UNSUPPORTED, H3_ERR_WORKSPACE,
 *         H3_ERR_MISALIGNED, H3_ERR_CUDA. */
H3_API h3_status h3_vsa_select(const void* q, const void* k, const int32_t grid[3],
                               const int32_t block[3], int32_t num_heads, int32_t head_dim,
                               int32_t topk, float softmax_scale, float* scores, int32_t* block_idx,
                               void* workspace, size_t workspace_bytes, h3_stream_t stream);

/* Workspace bytes of h3_vsa_attn_fwd (the key/value schedule); 0 for invalid sizes. */
H3_API size_t h3_vsa_attn_workspace_size(const int32_t grid[3], const int32_t block[3],
                                         int32_t num_heads, int32_t topk);

/* Token-level attention over the selected blocks: query i of block a attends, with one softmax,
 * to every key row of the blocks block_idx[h][a][0..topk) (rows inside the grid only).
 * q, k, v, o : device bf16 [T*H*W, num_heads, head_dim] (layout above); o gets every row.
 * lse        : device fp32 [num_heads, T*H*W] (natural log) or NULL.
 * block_idx  : device int32 [num_heads, nblk, topk], e.g. from h3_vsa_select; any order, ids
 *              distinct per list (a repeated id counts its keys twice).  An id outside [0, nblk)
 *              is replaced by block 0 and recorded as H3_ERR_BAD_BLOCK_INDEX.
 * softmax_scale: <= 0 selects 1/sqrt(head_dim).
 * workspace  : device, >= h3_vsa_attn_workspace_size() bytes, 16-byte aligned; overwritten.
 * Query blocks 2p and 2p + 1 share a 128-row tile, and each step of the tile loads two key blocks.
 * A first kernel writes each pair's steps into the workspace. When both lists are in ascending
 * order (as h3_vsa_select writes them), a block both query blocks selected serves both in one
 * step, so a pair sharing s blocks takes ceil(s/2) + topk - s steps instead of topk. Lists in any
 * other order take topk steps. The result is the same either way, up to summation order.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_UNSUPPORTED, H3_ERR_WORKSPACE,
 *         H3_ERR_MISALIGNED, H3_ERR_CUDA; device-side H3_ERR_BAD_BLOCK_INDEX / H3_ERR_TIMEOUT. */
H3_API h3_status h3_vsa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const int32_t grid[3], const int32_t block[3], int32_t num_heads,
                                 int32_t head_dim, const int32_t* block_idx, int32_t topk,
                                 float softmax_scale, void* workspace, size_t workspace_bytes,
                                 h3_stream_t stream);

/* ---- Continuation window ---------------------------------------------------------------------
 * [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section "Crossing
 * the time boundary": the last 7 latent video frames and the audio tail cut on the global 40 Hz
 * boundary are taken from the previous window's latents (step 1); the DiT sequence concatenates
 * (1) text / reference rows, (2) the audio tail, (3) the video tail, (4) new audio noise,
 * (5) new video noise, and only (4) and (5) are updated by the denoising steps (step 2); every
 * row's time coordinate is shifted by s * 40 / 24 before RoPE (step 3, h3_rope_apply with
 * start_frames = {s}); afterwards the new samples overlapping the tails are discarded and the
 * rest is appended to the clip.
 *
 * Readings where the pages leave a step open: a latent frame spans frames_per_latent video frames
 * at 24 FPS and audio latents are 40 Hz rows; the new window starts where the video tail starts,
 * g0 = clip_video_frames - tail_frames latent frames, s = g0 * frames_per_latent; the audio tail
 * starts at row floor(s * 40 / 24) (the row holding time s / 24 s); positions are local to the new
 * window (the tails and the new rows both start at t = 0); every group shares one row size; the
 * whole sequence is one attention segment.  Rows of every tensor are row_bytes bytes, contiguous;
 * video latents are frames of frame_h x frame_w rows in row-major (t, h, w) order. */
typedef struct {
  int32_t text_rows;           /* group 1 */
  int32_t clip_video_frames;   /* latent frames in the clip so far (>= tail_frames) */
  int32_t clip_audio_rows;     /* 40 Hz audio rows in the clip so far */
  int32_t frame_h, frame_w;    /* latent grid of one video frame */
  int32_t new_video_frames;    /* latent frames the new window samples (>= tail_frames) */
  int32_t new_audio_rows;      /* audio rows the new window samples (>= the audio tail) */
  int32_t tail_frames;         /* video tail, 7 on the pages */
  int32_t frames_per_latent;   /* video frames (24 FPS) per latent frame */
} h3_continuation_cfg;

typedef struct {
  int32_t tail_start;          /* g0: first latent frame of the video tail */
  int32_t start_frame;         /* s = g0 * frames_per_latent (the RoPE start frame) */
  int32_t audio_cut;           /* first audio row of the audio tail, min(floor(s*40/24), clip rows) */
  int32_t group_rows[5];       /* rows of the five groups in packed order */
  int32_t group_offset[6];     /* exclusive prefix of group_rows */
  int32_t num_rows;            /* rows of the packed sequence */
  int32_t keep_video_from;     /* first new latent frame appended (= tail_frames) */
  int32_t keep_audio_from;     /* first new audio row appended (= clip_audio_rows - audio_cut) */
  int32_t out_video_frames;    /* clip length after the append */
  int32_t out_audio_rows;
} h3_continuation_plan;

/* Host-only index math of a continuation window (no device work).
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG (a negative size, a clip or new window shorter than the
 * tail, new audio shorter than the audio tail, more than INT32_MAX rows). */
H3_API h3_status h3_continuation_make_plan(const h3_continuation_cfg* cfg, h3_continuation_plan* plan);

/* Pack the five groups: rows [num_rows, row_bytes], positions fp32 [num_rows, 3] (t, h, w; local
 * to the new window), tags uint8 [num_rows] (H3_TAG_*), target uint8 [num_rows] (1 on groups 4
 * and 5).  text [text_rows], clip_video [clip_video_frames * frame_h * frame_w], clip_audio
 * [clip_audio_rows], new_video [new_video_frames * frame_h * frame_w], new_audio [new_audio_rows]
 * rows; a source with no rows may be NULL.  row_bytes a positive multiple of 16; row pointers
 * 16-byte aligned, pos 4-byte aligned.  rows must not overlap a source.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_MISALIGNED, H3_ERR_CUDA. */
H3_API h3_status h3_continuation_pack(const h3_continuation_cfg* cfg, const void* text,
                                      const void* clip_video, const void* clip_audio,
                                      const void* new_video, const void* new_audio,
                                      int32_t row_bytes, void* rows, float* pos, uint8_t* tag,
                                      uint8_t* target, h3_stream_t stream);

/* Overlap discard and append: new video frames [tail_frames, new_video_frames) are written after
 * the clip's clip_video_frames frames, new audio rows [keep_audio_from, new_audio_rows) after its
 * clip_audio_rows rows; the clip's existing rows are untouched.  clip_video / clip_audio are the
 * clip's buffers with room for out_video_frames frames / out_audio_rows rows (capacities in rows
 * are checked).  Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_MISALIGNED, H3_ERR_CUDA. */
H3_API h3_status h3_continuation_append(const h3_continuation_cfg* cfg, const void* new_video,
                                        const void* new_audio, int32_t row_bytes, void* clip_video,
                                        int64_t clip_video_capacity_rows, void* clip_audio,
                                        int64_t clip_audio_capacity_rows, h3_stream_t stream);

/* Target-only update: dst row i = src row i where mask[i] != 0, other rows untouched.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG, H3_ERR_MISALIGNED, H3_ERR_CUDA. */
H3_API h3_status h3_masked_row_update(void* dst, const void* src, const uint8_t* mask,
                                      int32_t num_rows, int32_t row_bytes, h3_stream_t stream);

/* ---- Window-aligned sequence parallelism: host-side plan ------------------------------------
 * [H3-fast] "window attention across GPUs", "Window-aligned SP": whole windows (all heads) are the
 * unit given to a GPU, so window attention stays local; regular and half-shifted layers
 * alternate, and at each switch an all-to-all moves tokens to the owners of the new windows;
 * cropped edge windows have unequal sizes, so windows are dealt out by token count, not by count.
 * These calls do the integer planning only (host, no device work, no collective): the caller
 * moves the rows with its own all-to-all.  Windows and shifts are as for h3_window_count. */

/* Owner rank of every window of one layer: windows by size descending (ties: lower id) each go to
 * the rank with the fewest tokens so far (ties: lower rank).
 * window_rank: int32 [h3_window_count()] out; rank_tokens: int64 [world] out or NULL.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG. */
H3_API h3_status h3_sp_assign_windows(const int32_t grid[3], const int32_t win[3],
                                      const int32_t shift[3], int32_t world, int32_t* window_rank,
                                      int64_t* rank_tokens);

/* Tokens each rank owns under a window -> rank map of one layer.
 * rank_tokens: int64 [world] out.  Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG. */
H3_API h3_status h3_sp_rank_tokens(const int32_t grid[3], const int32_t win[3],
                                   const int32_t shift[3], const int32_t* window_rank,
                                   int32_t world, int64_t* rank_tokens);

/* A rank's local row order in one layer: the original (row-major) index of each token it owns,
 * its windows ascending and tokens row-major inside (the single-GPU packed order restricted to
 * the rank).  order: int32 [rank_tokens[rank]] out (order_capacity entries available).
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG (bad geometry, rank or owner, or capacity too small). */
H3_API h3_status h3_sp_layer_order(const int32_t grid[3], const int32_t win[3],
                                   const int32_t shift[3], const int32_t* window_rank,
                                   int32_t world, int32_t rank, int32_t* order,
                                   int64_t order_capacity);

/* The all-to-all of a switch from layer `from` (shift_from, owners rank_from) to layer `to`,
 * as seen by `rank`:
 *   send_counts [world] out: rows this rank sends to each rank;
 *   send_index  [sum send_counts] out: the rows of this rank's `from` layout to send, grouped by
 *               destination rank ascending, each group in the destination's `to` order;
 *   recv_counts [world] out: rows received from each rank;
 *   recv_position [sum recv_counts] out: for the rows as they arrive (grouped by source rank
 *               ascending, each group in this rank's `to` order), their row in this rank's `to`
 *               layout.
 * Gather by send_index, all-to-all with these counts, scatter to recv_position: the rank then
 * holds its `to` windows in the order of h3_sp_layer_order.
 * Errors: H3_ERR_NULL, H3_ERR_INVALID_ARG. */
H3_API h3_status h3_sp_exchange_plan(const int32_t grid[3], const int32_t win[3],
                                     const int32_t shift_from[3], const int32_t* rank_from,
                                     const int32_t shift_to[3], const int32_t* rank_to,
                                     int32_t world, int32_t rank, int64_t* send_counts,
                                     int32_t* send_index, int64_t* recv_counts,
                                     int32_t* recv_position);

/* ---- Testing hooks of the timeout path (no page counterpart) --------------------------------
 * Every wait between the warps of an attention kernel (h3_varlen_attn_fwd, its no-alloc form,
 * h3_window_attn_fwd, h3_vsa_attn_fwd) is bounded.  A wait that runs out records H3_ERR_TIMEOUT;
 * the kernel then waits (always with the default 2 s limit) for the copies and matrix products it
 * has already issued, releases its tensor memory and returns, and every later attention launch
 * leaves at once until h3_get_device_error() clears the error.  Outputs of a launch that timed
 * out are unspecified (partly written).  These two process-wide settings let tests drive that
 * path; they apply to attention launches issued after the call. */

/* Limit, in nanoseconds, of the pipeline waits; 0 restores the default of 2 s.  Returns the limit
 * in force before the call. */
H3_API uint64_t h3_set_wait_limit_ns(uint64_t nanoseconds);

/* The key/value loader of each attention CTA issues at most `tiles` tiles and then stops, as if
 * it had stalled, so the waits of the warps that consume them run out; negative (the default)
 * restores normal operation.  Nothing is read or written out of bounds and every wait still ends
 * by its limit.  Returns the previous setting. */
H3_API int32_t h3_debug_stall_loads(int32_t tiles);

/* Synchronises `stream`, returns the first device-side error recorded on the current device
 * since the last call (H3_OK if none) and clears it. */
H3_API h3_status h3_get_device_error(h3_stream_t stream);

/* Static description of a status code. */
H3_API const char* h3_status_string(h3_status status);

/* Library ABI version (major * 100 + minor). */
H3_API int32_t h3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H_ */
