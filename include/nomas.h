/*
 * nomas.h -- C ABI of the B300 (sm_103a) segment-causal attention library (libnomas.so).
 *
 * The library implements the hot path of a segment-autoregressive MMDiT video world
 * model as the Hy-Nomas pages describe it:
 *   * 3D RoPE on Q/K, head dim 128 split [16, 56, 56] over (t, h, w), theta 256
 *     (comfyui-wiki news, section "模型内部", architecture table);
 *   * an INT8 "lifelong" KV cache of every earlier segment (huaweicloud blog, section 2.1:
 *     each segment's text/video K,V are cached and passed to the next segment;
 *     comfyui-wiki, section "单张 4090 配置": cached K/V stored INT8, attention in BF16);
 *   * segment-causal attention: a segment attends to the cache of every earlier segment,
 *     never to a later one (comfyui-wiki, section "一个世界，分段生成");
 *   * a temporal_context gather that packs 18 selected history latent frames into a
 *     contiguous device history (comfyui-wiki, section "单张 4090 配置").
 *
 * Conventions for every call
 *   * Pointers marked (device) are CUDA device pointers owned by the caller; the library
 *     never frees them and keeps none of them after the call returns.  Pointers marked
 *     (host) are read during the call only.
 *   * head_dim is 128.  Every device pointer must be 16-byte aligned; token strides are
 *     given in elements and must be multiples of 8 (16 bytes of BF16).
 *   * All argument checks run on the host before anything is enqueued; on any error
 *     nothing is written and nothing is launched.  nomas_last_error() then describes it.
 *   * Work is enqueued asynchronously on `stream`.  Device-side failures (a bounded wait
 *     that gave up) are reported by nomas_stream_check().
 *   * No call allocates device memory on the hot path: the attention workspace comes from
 *     the caller (see nomas_seg_attn_workspace_size).  Only nomas_rope_tables_create
 *     allocates (its tables), once.
 *   * The library is not re-entrant across threads for one stream; distinct streams are
 *     independent.  C++ exceptions never cross this boundary.
 */
#ifndef NOMAS_H
#define NOMAS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NOMAS_HEAD_DIM 128
#define NOMAS_MAX_SEGMENTS 64        /* current segments per nomas_seg_attn call */
#define NOMAS_MAX_GATHER_FRAMES 2048 /* frames per nomas_kv_gather_context call */
#define NOMAS_MAX_ATTN_HEADS 4096    /* heads per nomas_seg_attn call */
#define NOMAS_MAX_CAMERA_TOKENS 128  /* camera tokens per nomas_camera_cross_attn call */

typedef enum {
    NOMAS_OK = 0,
    NOMAS_EINVAL = 1,        /* a bad argument (null, misaligned, out of range) */
    NOMAS_ECAPACITY = 2,     /* the destination cache is too small */
    NOMAS_EUNSUPPORTED = 3,  /* valid but not supported here (head_dim != 128, too many segments) */
    NOMAS_ECUDA = 4,         /* a CUDA runtime/driver call failed */
    NOMAS_ETIMEOUT = 5,      /* a kernel's bounded wait gave up (reported by nomas_stream_check) */
    NOMAS_ERANGE = 6         /* input magnitudes beyond what the fp32 softmax represents (reported by
                                nomas_stream_check; the call's outputs are then unspecified) */
} nomas_status;

/* One segment's token layout: T*grid_h*grid_w video tokens in (t, h, w) row-major order,
 * t from t0 (global latent frame index), h in [0, grid_h), w in [0, grid_w); then n_text
 * text tokens, which carry no position and are never rotated. */
typedef struct {
    int32_t t0, T, grid_h, grid_w, n_text;
} nomas_segment;

/* INT8 KV cache (device memory owned by the caller).
 *   k, v          : int8  [heads][capacity][head_dim]  (head-major)
 *   k_scale, v_sc.: fp32  [heads][capacity]
 *   length        : valid tokens, rows [0, length) of every head
 * Row (h, j) dequantises to code * scale.  capacity must be a multiple of 4. */
typedef struct {
    int8_t *k, *v;
    float *k_scale, *v_scale;
    int64_t capacity, length;
    int32_t heads, head_dim;
} nomas_kv_cache;

/* Opaque RoPE cos/sin tables (device-resident, created once). */
typedef struct nomas_rope_tables nomas_rope_tables;

/* ------------------------------------------------------------------ RoPE tables
 * comfyui-wiki news, architecture table: 3D RoPE sizes [16, 56, 56], theta 256.
 * For axis a with d_a = split[a] channels, pair i in [0, d_a/2) rotates by
 * pos * theta^(-2i/d_a); cos/sin are computed in double on the host and rounded once to
 * fp32, for pos in [0, max_t) / [0, max_h) / [0, max_w).  split must be even numbers
 * summing to 128, each a multiple of 8.  *out receives the handle (free with destroy). */
nomas_status nomas_rope_tables_create(float theta, const int32_t split[3], int32_t max_t,
                                      int32_t max_h, int32_t max_w, nomas_rope_tables **out);
void nomas_rope_tables_destroy(nomas_rope_tables *tables);
/* Copies the host copy of axis `axis` (0 = t, 1 = h, 2 = w) into cos_out/sin_out (host,
 * [max_pos][split[axis]/2] fp32 each).  For checking the tables; no GPU work. */
nomas_status nomas_rope_tables_read(const nomas_rope_tables *tables, int32_t axis,
                                    float *cos_out, float *sin_out);

/* ----------------------------------------------------------------------- rope3d
 * Rotates the video tokens of one segment: y = RoPE(x), BF16 in, BF16 out.
 * Pair (x0, x1) -> (x0*c - x1*s, x0*s + x1*c), each product and sum rounded to fp32
 * (no FMA), the result rounded to BF16 (nearest-even).  Text tokens are copied.
 *   x, y       : (device) bf16 [n][heads][128], n = seg tokens, token stride row_stride
 *                elements (>= heads*128); y may equal x (in place), otherwise they must
 *                not overlap.
 * Errors: EINVAL on null/misaligned pointers, a position outside the tables. */
nomas_status nomas_rope3d(const void *x_bf16, void *y_bf16, int64_t row_stride,
                          const nomas_segment *seg, int32_t heads,
                          const nomas_rope_tables *tables, cudaStream_t stream);

/* ------------------------------------------------------------ append + quantise
 * Appends one finished segment's K/V to the INT8 cache (huaweicloud blog 2.1; comfyui-wiki
 * "单张 4090 配置").  For token k and head h:
 *   K row: BF16(RoPE(K)) for video tokens (text: K unchanged), then quantised;
 *   V row: quantised without rotation.
 * Quantisation of a 128-value row x (fp32 of the BF16 values): a = max|x|;
 *   scale = a / 127 (fp32, IEEE division); a == 0 -> scale 0, codes 0;
 *   else code = clamp(round_half_even(x / scale), -127, 127) (fp32 IEEE quotient).
 * Rows are written at cache positions [length, length + n); on success cache->length += n.
 *   k, v : (device) bf16 [n][heads][128], token stride row_stride elements.
 * Errors: ECAPACITY if length + n > capacity (nothing written); EINVAL on a heads mismatch
 * or bad pointers; EUNSUPPORTED if head_dim != 128. */
nomas_status nomas_kv_append_quant(nomas_kv_cache *cache, const void *k_bf16, const void *v_bf16,
                                   int64_t row_stride, const nomas_segment *seg,
                                   const nomas_rope_tables *tables, cudaStream_t stream);

/* ------------------------------------------------------ temporal_context gather
 * Packs selected frames of an archive cache into a contiguous history (comfyui-wiki,
 * "单张 4090 配置": GPU history limited to temporal_context-sampled latent frames).
 *   frame_token_offset : (host) [n_archive_frames] first archive token of each frame
 *   frames             : (host) [n_frames] selected frame indices, strictly increasing
 *   index_map          : (device, nullable) int32 [n_frames * tokens_per_frame]
 * Packed token j = archive token frame_token_offset[frames[j / tpf]] + j % tpf; its codes
 * and scales (all heads) are copied to dst row j, index_map[j] receives that archive
 * token.  dst rows [0, n) are written and, on success, dst->length = n = n_frames *
 * tokens_per_frame; on any error dst->length is left unchanged.
 * Errors: EINVAL (unsorted/out-of-range frames, a source row outside archive->length,
 * heads mismatch), ECAPACITY (n > dst->capacity), EUNSUPPORTED (n_frames > 2048). */
nomas_status nomas_kv_gather_context(const nomas_kv_cache *archive, const int32_t *frame_token_offset,
                                     int32_t n_archive_frames, int32_t tokens_per_frame,
                                     const int32_t *frames, int32_t n_frames, nomas_kv_cache *dst,
                                     int32_t *index_map, cudaStream_t stream);

/* ------------------------------------------ temporal_context gather, host archive
 * The same gather with the archive in pinned system memory, as the single-GPU design of the
 * pages keeps the history beyond the temporal_context frames off the GPU (comfyui-wiki,
 * "单张 4090 配置"; huaweicloud blog, 三、部署实战: the older history lives on the host).
 *   archive            : (host, pinned: cudaHostAlloc or cudaHostRegister) codes and scales,
 *                        same layout as a device cache
 *   dst, index_map     : (device) as for nomas_kv_gather_context
 * The copy engines move the rows (one 2-D copy per array and per run of frames that are
 * consecutive in the archive, all heads at once), so on a stream of its own the gather overlaps
 * kernels on other streams; only the optional index map uses a kernel.  Results are identical
 * to nomas_kv_gather_context.  Errors: those of nomas_kv_gather_context, and EINVAL if an
 * archive buffer is not pinned host memory.  Every check runs before the first copy is
 * enqueued; only a copy the CUDA runtime refuses after others were enqueued (NOMAS_ECUDA) can
 * leave rows of dst partly overwritten, with dst->length unchanged. */
nomas_status nomas_kv_gather_context_host(const nomas_kv_cache *archive, const int32_t *frame_token_offset,
                                          int32_t n_archive_frames, int32_t tokens_per_frame,
                                          const int32_t *frames, int32_t n_frames, nomas_kv_cache *dst,
                                          int32_t *index_map, cudaStream_t stream);

/* ----------------------------------------------------- segment-causal attention
 * comfyui-wiki news, "一个世界，分段生成": the segment being denoised attends to the K/V of
 * every earlier segment (the INT8 history, always visible) and, within the current call,
 * query i of segment s sees the current keys of segments 0..s (bidirectional inside s).
 *   O_i = sum_j softmax_j(q_i . k_j * softmax_scale) v_j
 * History keys/values are the INT8 codes times their scales.
 * Arithmetic: the tensor-core operands are FP16, each operand block multiplied by an exact power of
 * two chosen from its largest magnitude so that the block's maximum lies in [2^14, 2^15): a query
 * row by its own factor, the current K and V of a head by one factor each, the head's history K
 * and V (code * scale, formed in fp32) by one factor each.  Every value within 2^28 of its block's
 * maximum is then a normal FP16 number (11 significant bits; BF16 inputs carry 8, so they convert
 * exactly), and the factors are undone exactly in fp32: in the softmax multiplier for Q and K, in
 * the output for V.  QK^T and PV run with fp32 accumulation, P is FP16, the online softmax is fp32.
 * This holds for any finite BF16 inputs, with two limits reported as NOMAS_ERANGE by
 * nomas_stream_check (the output is then unspecified): a query row whose largest possible score
 * |q|max * |k|max * softmax_scale exceeds about 1e34, and a head whose current and history V maxima
 * differ by more than 2^70.  Non-finite inputs give undefined results.
 * The call first writes these FP16 operands into the workspace (an HBM-bound pass over Q, K, V
 * and the history), then runs the attention kernel on them.  A caller that attends to the same
 * history several times (the denoising steps of one segment) can stage the history once with
 * nomas_seg_attn_stage_history and call nomas_seg_attn_staged instead.
 *   q, k_cur, v_cur : (device) bf16 [Lq][heads][128], token stride row_stride elements
 *                     (q and k_cur already rotated by nomas_rope3d)
 *   q_seg_offsets   : (host) int32 [n_seg + 1], 0 = off[0] <= ... <= off[n_seg] = Lq
 *   history         : (nullable) INT8 cache, rows [0, length) used; may have length 0
 *   softmax_scale   : 0 -> 1/sqrt(128)
 *   out             : (device) bf16 [Lq][heads][128], token stride heads*128
 *   lse             : (device, nullable) fp32 [heads][Lq], natural-log log-sum-exp
 *   workspace       : (device) at least nomas_seg_attn_workspace_size(Lq, Lh, heads) bytes;
 *                     contents need not be initialised and are overwritten: the staged FP16
 *                     operands ((3 Lq + 2 Lh) x heads x 256 bytes), the history scale maxima, the
 *                     split-KV partials when the key range is split across CTAs, the query-row
 *                     exponents (Lq x heads bytes) and the current K/V maxima.
 * Deterministic: no floating-point atomics; a fixed reduction order for any given shapes.
 * Errors: EINVAL (bad offsets/pointers/strides, heads mismatch), EUNSUPPORTED
 * (n_seg > 64 or heads > 4096), EINVAL if the workspace is too small. */
nomas_status nomas_seg_attn(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16,
                            int64_t row_stride, int32_t heads, const int32_t *q_seg_offsets,
                            int32_t n_seg, const nomas_kv_cache *history, float softmax_scale,
                            void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);
/* Workspace bytes nomas_seg_attn needs for these sizes; host-only.  0 if lq <= 0 or the sizes are
 * beyond what nomas_seg_attn accepts (Lq or Lh of 2^30 or more, heads outside 1..4096,
 * 2 x heads x Lh of 2^31 or more). */
size_t nomas_seg_attn_workspace_size(int64_t lq, int64_t lh, int32_t heads);

/* ------------------------------------------- segment-causal attention, staged history
 * The history does not change while a segment is denoised (comfyui-wiki news, "一个世界，分段生成":
 * each segment attends to the fixed cache of the earlier ones; its several Euler steps see the
 * same history).  nomas_seg_attn_stage_history writes the history's FP16 operands once, and
 * nomas_seg_attn_staged attends to them from every step, so the per-step work is the current
 * segment's staging plus the attention kernel.
 *
 * A staged history (device memory owned by the caller):
 *   data     : (device) nomas_staged_history_size(capacity, heads) bytes, 16-byte aligned: the
 *              per-head maxima of the k and v row scales, then FP16 K and V [heads][capacity][128]
 *   bytes    : size of data
 *   capacity : rows per head the buffer holds
 *   length   : rows staged (written by nomas_seg_attn_stage_history)
 *   heads    : heads of the history it holds
 * The staged copy is a snapshot: after the INT8 cache changes (an append, a gather) it must be
 * staged again; the caller owns that validity. */
typedef struct {
    void *data;
    size_t bytes;
    int64_t capacity, length;
    int32_t heads;
} nomas_staged_history;
/* Bytes of a staged history of `capacity` rows per head (0 if either argument is <= 0). */
size_t nomas_staged_history_size(int64_t capacity, int32_t heads);
/* Stages rows [0, history->length) of the INT8 history into `staged` (same operands, bit for bit,
 * as nomas_seg_attn stages inside its workspace) and sets staged->length.  staged->heads must
 * equal history->heads.  Errors: EINVAL (cache, buffer, heads), ECAPACITY (length > capacity),
 * EUNSUPPORTED (heads x rows >= 2^30); nothing is written on error. */
nomas_status nomas_seg_attn_stage_history(const nomas_kv_cache *history, nomas_staged_history *staged,
                                          cudaStream_t stream);
/* nomas_seg_attn over a staged history: same arguments, results and errors, with `history` a
 * staged history (nullable; length 0 means none) and a workspace of
 * nomas_seg_attn_staged_workspace_size(Lq, history->length, heads) bytes (the history's share of
 * nomas_seg_attn's workspace is the staged buffer).  Results are bit-identical to nomas_seg_attn
 * on the INT8 history that was staged. */
nomas_status nomas_seg_attn_staged(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16,
                                   int64_t row_stride, int32_t heads, const int32_t *q_seg_offsets,
                                   int32_t n_seg, const nomas_staged_history *history, float softmax_scale,
                                   void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream);
/* Workspace bytes nomas_seg_attn_staged needs; host-only, 0 on the same conditions as
 * nomas_seg_attn_workspace_size. */
size_t nomas_seg_attn_staged_workspace_size(int64_t lq, int64_t lh, int32_t heads);

/* ------------------------------------- segment-causal attention, no allocation
 * The Hy-Nomas pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory where they run attention.  Examples: a serving process whose
 * framework allocator has already reserved the device memory (cudaMalloc would fail or
 * fragment it), or a latency-critical loop where cudaMalloc/cudaFree would synchronise the
 * device.  nomas_seg_attn needs a caller workspace for its staged operands and split-KV
 * partials; this variant takes that scratch from one fixed device array inside the library
 * instead, and allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 * Arguments, results and errors are those of nomas_seg_attn without the workspace.  The
 * caller still owns and passes q, k_cur, v_cur, out and lse.
 *   * Limit: the scratch holds NOMAS_NOALLOC_SCRATCH_BYTES (32 MiB).  A call whose
 *     nomas_seg_attn_workspace_size(Lq, Lh, heads) exceeds it returns NOMAS_ECAPACITY with a
 *     message (nomas_last_error) and launches nothing; use nomas_seg_attn with a workspace.
 *   * The array is held by every GPU that loads the library until the process exits.
 *   * Set-up: the first call on each device, with that device current, looks up the array's
 *     device address (cudaGetSymbolAddress; NOMAS_ECUDA if that fails).  Make that first call
 *     before any stream capture.
 *   * Every call shares the one array and leaves its contents behind; each call writes every
 *     staged operand, partial and exponent it later reads, and resets the per-head maxima it
 *     accumulates (cudaMemsetAsync, which allocates nothing), so nothing else has to start at
 *     zero.  Calls whose kernels overlap on the GPU (other streams, other threads) race on the
 *     array: serialise them. */
#define NOMAS_NOALLOC_SCRATCH_BYTES (32u << 20)
nomas_status nomas_seg_attn_noalloc(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16,
                                    int64_t row_stride, int32_t heads, const int32_t *q_seg_offsets,
                                    int32_t n_seg, const nomas_kv_cache *history, float softmax_scale,
                                    void *out_bf16, float *lse, cudaStream_t stream);

/* ------------------------------------------- QKV projection with fused 3D RoPE
 * The linear layer that produces a block's Q, K and V from its hidden states, with INT8
 * weights and BF16 activations (comfyui-wiki news, 模型内部: hidden size 2,048 = 16 heads x 128;
 * 单张 4090 配置: DiT weights stored INT8, linear layers computed in BF16), followed by the 3D RoPE
 * of Q and K exactly as nomas_rope3d applies it:
 *   p[l, n] = BF16( w_scale[n] * sum_k x[l, k] * w_codes[n, k] )   (fp32 accumulation)
 *   qkv[l, 0, h, :] = RoPE(p[l, h*128 : h*128+128]),  qkv[l, 1, h, :] = RoPE(p[l, (H+h)*128 : ...]),
 *   qkv[l, 2, h, :] = p[l, (2H+h)*128 : ...]   (RoPE of video tokens only, as nomas_rope3d)
 *   x        : (device) bf16 [L][hidden], token stride x_row_stride elements (L = seg tokens)
 *   w_codes  : (device) int8 [3*heads*128][hidden], output channel n's codes (row n)
 *   w_scale  : (device) fp32 [3*heads*128], output channel n's scale
 *   qkv      : (device) bf16 [L][3][heads][128], token stride out_row_stride elements
 *   workspace: (device) nomas_qkv_project_workspace_size(heads, hidden) bytes (the codes as
 *              BF16, exact); contents need not be initialised.
 * heads must be even (at most 4096) and hidden a multiple of 64 (at most 65536).  Errors:
 * EINVAL (pointers, strides, workspace, positions outside the tables), EUNSUPPORTED (heads,
 * hidden). */
nomas_status nomas_qkv_project_rope(const void *x_bf16, int64_t x_row_stride, int32_t hidden,
                                    const int8_t *w_codes, const float *w_scale, int32_t heads,
                                    const nomas_segment *seg, const nomas_rope_tables *tables,
                                    void *qkv_bf16, int64_t out_row_stride, void *workspace,
                                    size_t workspace_bytes, cudaStream_t stream);
/* Workspace bytes nomas_qkv_project_rope needs (0 if heads or hidden <= 0); host-only. */
size_t nomas_qkv_project_workspace_size(int32_t heads, int32_t hidden);

/* nomas_qkv_project_rope plus the append of the segment's K and V to the INT8 cache in the same
 * kernel, for the segment's final denoising step (the cached K/V of a finished segment, [huawei]
 * 2.1; stored INT8 per [comfyui] 单张 4090 配置).  The cache rows written are exactly those
 * nomas_kv_append_quant(cache, k, v, seg) writes when given the projection's K and V before the
 * RoPE (it rotates K itself, and the fused path rotates, rounds to BF16 and quantises the same
 * values): codes and scales bit for bit, at rows cache->length .. cache->length + L - 1, and
 * cache->length advances by L when the work is enqueued.  If nomas_stream_check later reports
 * NOMAS_ETIMEOUT for this call (its kernel gave up a bounded wait), those rows were not written:
 * the caller must set cache->length back by L before the cache is used again.  Arguments as
 * nomas_qkv_project_rope; cache->heads must equal heads.
 * Errors: those of nomas_qkv_project_rope, EINVAL for a NULL or malformed cache, ECAPACITY if
 * length + L > capacity (nothing written). */
nomas_status nomas_qkv_project_rope_append(const void *x_bf16, int64_t x_row_stride, int32_t hidden,
                                           const int8_t *w_codes, const float *w_scale, int32_t heads,
                                           const nomas_segment *seg, const nomas_rope_tables *tables,
                                           void *qkv_bf16, int64_t out_row_stride, void *workspace,
                                           size_t workspace_bytes, nomas_kv_cache *cache, cudaStream_t stream);

/* ------------------------------------------------------------ camera conditioning
 * comfyui-wiki news, 相机控制作为一等输入: a trajectory file gives camera-to-world matrices
 * c2ws [N, 4, 4] (and intrinsics, not used here); the extrinsics are normalised, grouped by four
 * video frames and each group flattened to a 64-value input, which the video tokens query
 * through a cross-attention in every dual-stream block (模型内部 table, 相机条件 row); the
 * scales trajectory_translation_scale and trajectory_rotation_scale default to 1.0 and 2.5.
 *
 * Camera tokens: with the first frame as reference, for every frame i
 *   E_i = [ rotation_scale * R0^T R_i | translation_scale * R0^T (t_i - t0) ; 0 0 0 1 ]
 * (the rigid inverse of c2w[0] times c2w[i], then the two scales), in fp32;
 * tokens[g][16 j + 4 r + c] = E_{4g+j}[r][c] for j, r, c in 0..3.
 *   c2w    : (device) fp32 [n_frames][4][4] row-major (R_i = rows 0-2, columns 0-2; t_i = column
 *            3); the bottom rows are not read.  16-byte aligned.
 *   tokens : (device) fp32 [n_frames / 4][64], 16-byte aligned, not overlapping c2w.
 * n_frames must be a positive multiple of 4 (at most 2^24); the scales must be finite.
 * Errors: EINVAL (pointers, alignment, n_frames, scales); nothing is written on error. */
nomas_status nomas_camera_tokens(const float *c2w, int32_t n_frames, float translation_scale,
                                 float rotation_scale, float *tokens, cudaStream_t stream);

/* Camera cross-attention: every video-token query attends to every camera token, per head:
 *   out[l, h, :] = sum_j softmax_j( q[l, h, :] . k[j, h, :] * scale ) v[j, h, :]
 * (no mask, no positions; scale = softmax_scale, or 1/sqrt(128) if softmax_scale is 0).
 * The camera tokens' K and V come from the block's embedding and projection of the tokens
 * nomas_camera_tokens builds (weights of the model, applied by the caller).
 *   q    : (device) bf16 [lq][heads][128], token stride q_row_stride elements
 *   k, v : (device) bf16 [n_cam][heads][128], token stride cam_row_stride elements
 *   out  : (device) bf16 [lq][heads][128], token stride out_row_stride elements; may be q
 *          itself (same stride: each (128-token, head) tile is read before it is written), must
 *          not overlap k or v.
 * Strides are multiples of 8 and at least heads*128; pointers 16-byte aligned.
 * Limits: 1 <= n_cam <= NOMAS_MAX_CAMERA_TOKENS, heads <= NOMAS_MAX_ATTN_HEADS,
 * ceil(lq / 128) * heads < 2^31.  lq = 0 is a no-op.  Arithmetic: q.k in BF16 tensor-core
 * products with fp32 accumulation, probabilities rounded to FP16, V in FP16 after an exact
 * multiplication by a power of two per head that puts the head's max |v| in [2^14, 2^15) (every
 * BF16 value within 2^28 of it converts exactly; the factor is undone in fp32), fp32
 * accumulation, BF16 output.  Scores beyond the fp32 range (|q| |k| near 1e18 and above) are
 * reported as NOMAS_ERANGE by nomas_stream_check, the output then unspecified.  Errors: EINVAL
 * (pointers, strides, scale, n_cam < 1), EUNSUPPORTED (n_cam, heads or tile count over the
 * limits). */
nomas_status nomas_camera_cross_attn(const void *q_bf16, int64_t q_row_stride, int32_t lq, int32_t heads,
                                     const void *k_cam_bf16, const void *v_cam_bf16,
                                     int64_t cam_row_stride, int32_t n_cam, float softmax_scale,
                                     void *out_bf16, int64_t out_row_stride, cudaStream_t stream);

/* ----------------------------------------------------------------- diagnostics
 * Synchronises `stream`, then reads and clears the library's device status word.
 * Returns ETIMEOUT if a kernel gave up a bounded wait since the last check, ECUDA if the
 * synchronisation failed, OK otherwise. */
nomas_status nomas_stream_check(cudaStream_t stream);
const char *nomas_status_string(nomas_status status);
/* Message describing the last failed call on this thread ("" if none). */
const char *nomas_last_error(void);
/* Library version string. */
const char *nomas_version(void);

/* Testing hook for failure detection without a GPU fault.  what = 1 arms the next
 * nomas_seg_attn launch (from any thread) to withhold its Q load: every CTA's bounded
 * waits then give up after about a second, the kernel records NOMAS_ETIMEOUT in the status
 * word (read and cleared by nomas_stream_check), lets the copies it already issued land,
 * frees its tensor memory and exits without writing `out`.  what = 0 disarms. */
void nomas_debug_inject(int32_t what);

/* Testing hook: which kernel variant the attention calls (nomas_seg_attn, nomas_seg_attn_staged,
 * nomas_seg_attn_noalloc) run from now on, from any thread.  variant = 1: one CTA per 256-row Q
 * block; 2: clusters of two CTAs on the two SMs of a pair (cta_group::2 MMAs over two Q blocks,
 * each SM loading half of every key tile); 0 (or any other value): chosen by the call's shape
 * (the pair variant for unsplit calls of at least 1e13 FLOP).  Both give results within the same
 * tolerance; the choice changes only the speed. */
void nomas_debug_attn_variant(int32_t variant);

#ifdef __cplusplus
}
#endif
#endif /* NOMAS_H */
