// internal.h -- host-side declarations shared by the libnomas translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nomas.h"

namespace nomas {

// Device-resident RoPE tables plus their host copies (for nomas_rope_tables_read).
struct RopeTablesImpl {
    int32_t split[3];
    int32_t max_pos[3];
    float *d_cos[3];  // device [max_pos][split/2]
    float *d_sin[3];
    float *h_cos[3];  // host copies
    float *h_sin[3];
    int device;
};

// Per-segment token layout passed to kernels by value.
struct SegDesc {
    int32_t t0, T, gh, gw, n_text;
    int32_t n_video;   // T * gh * gw
    int32_t n_tokens;  // n_video + n_text
};

struct RopeDev {
    const float *cos[3];
    const float *sin[3];
    int32_t max_pos[3];
};

// Replaces the calling thread's nomas_last_error() message.
void set_last_error(const char *msg);

// Library device status word (2 ints: code, where) for the current device.
int *device_status_word();

// Kernel launchers (return a CUDA error from the launch).
cudaError_t launch_rope3d(const void *x, void *y, int64_t row_stride, const SegDesc &seg, int32_t heads,
                          const RopeDev &rope, cudaStream_t stream);
cudaError_t launch_append_quant(const void *k, const void *v, int64_t row_stride, const SegDesc &seg,
                                int32_t heads, const RopeDev &rope, int8_t *ck, int8_t *cv, float *cks,
                                float *cvs, int64_t cap, int64_t length, cudaStream_t stream);
cudaError_t launch_index_map(const int32_t *src_frame_token, int32_t n_frames, int32_t tpf, int32_t *index_map,
                             cudaStream_t stream);
cudaError_t launch_gather(const nomas_kv_cache &src, const int32_t *src_frame_token, int32_t n_frames,
                          int32_t tpf, nomas_kv_cache &dst, int32_t *index_map, cudaStream_t stream);

struct AttnLaunch {
    const void *q, *k, *v;
    int64_t row_stride;
    int32_t heads;
    int32_t lq;
    int32_t n_seg;
    const int32_t *seg_off;      // host, n_seg + 1
    const void *hist_block;      // staged history (maxima header, FP16 K, V), or null when lh == 0
    int64_t hist_cap;            // rows per head of the staged history block
    int64_t lh;                  // history rows attended
    float softmax_scale;
    void *out;
    float *lse;
    void *workspace;             // the current operands, partials, Q exponents and maxima
    size_t part_off, qexp_off, max_off;  // offsets into the workspace (attn_workspace_layout)
    int32_t n_splits;
    int32_t fault;
    int32_t variant;             // 0: chosen by shape; 1: the single-CTA kernel; 2: the CTA-pair kernel
};
int32_t attn_num_splits(int64_t lq, int64_t lh, int32_t heads, int num_sms);
// The attention workspace, in this order: staged FP16 Q, K, V ([heads][lq][128] each); when the
// call stages the history itself, its staged-history block; the split-KV partials (fp32 O, then
// LSE); the per-row Q exponents (int8 [heads][lq]); the per-head maxima of the current K and V.
struct AttnWorkspace {
    size_t cur_bytes, hist_off, hist_bytes, part_off, part_bytes, qexp_off, qexp_bytes, max_off, max_bytes, total;
};
AttnWorkspace attn_workspace_layout(int64_t lq, int64_t lh, int32_t heads, int32_t n_splits, bool with_history);
// A staged-history block of cap_rows rows per head: a header with the per-head maxima of the k and
// v row scales (uint32 [2][heads], fp32 bit patterns), then FP16 K and V [heads][cap_rows][128].
size_t staged_history_header_bytes(int32_t heads);
size_t staged_history_bytes(int64_t cap_rows, int32_t heads);
// Stages rows [0, lh) of an INT8 history into `block` (cap_rows >= lh rows per head).
nomas_status launch_stage_history(const nomas_kv_cache &h, int64_t lh, void *block, int64_t cap_rows,
                                  cudaStream_t stream, char *err, size_t err_len);
nomas_status launch_seg_attn(const AttnLaunch &a, cudaStream_t stream, char *err, size_t err_len);

// The arguments of nomas_seg_attn and its variants (history: an INT8 cache the call stages
// itself, or staged: a history staged earlier; at most one is non-null).
struct SegAttnArgs {
    const char *what;
    const void *q, *k, *v;
    int64_t row_stride;
    int32_t heads;
    const int32_t *offs;
    int32_t n_seg;
    const nomas_kv_cache *history;
    const nomas_staged_history *staged;
    float softmax_scale;
    void *out;
    float *lse;
    cudaStream_t stream;
};
// Validates everything but the workspace (nothing launched; nomas_last_error set on failure);
// *lq and *lh receive the query and history row counts.
nomas_status seg_attn_check(const SegAttnArgs &a, int32_t *lq, int64_t *lh);
// Runs checked arguments with the given workspace (checked against the layout's size here).
nomas_status seg_attn_run(const SegAttnArgs &a, int32_t lq, int64_t lh, void *workspace, size_t workspace_bytes);

struct QkvLaunch {
    const void *x;          // bf16 [lq][hidden], token stride x_row_stride elements
    int64_t x_row_stride;
    int32_t hidden, heads, lq;
    const int8_t *w_codes;  // [3 * heads * 128][hidden]
    const float *w_scale;   // [3 * heads * 128]
    SegDesc seg;
    RopeDev rope;
    void *out;              // bf16 [lq][3][heads][128], token stride out_row_stride elements
    int64_t out_row_stride;
    void *workspace;        // qkv_project_workspace_bytes(heads, hidden)
    const nomas_kv_cache *cache;  // fused append of K and V at cache->length, or null
};
size_t qkv_project_workspace_bytes(int32_t heads, int32_t hidden);
nomas_status launch_qkv_project(const QkvLaunch &a, cudaStream_t stream, char *err, size_t err_len);

cudaError_t launch_camera_tokens(const float *c2w, int32_t n_frames, float translation_scale,
                                 float rotation_scale, float *tokens, cudaStream_t stream);
struct CamLaunch {
    const void *q;           // bf16 [lq][heads][128], token stride q_row_stride elements
    int64_t q_row_stride;
    int32_t lq, heads;
    const void *k, *v;       // bf16 [n_cam][heads][128], token stride cam_row_stride elements
    int64_t cam_row_stride;
    int32_t n_cam;
    float softmax_scale;     // 0: 1/sqrt(128)
    void *out;               // bf16 [lq][heads][128], token stride out_row_stride elements
    int64_t out_row_stride;
};
nomas_status launch_camera_xattn(const CamLaunch &a, cudaStream_t stream, char *err, size_t err_len);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
int device_sm_count();

}  // namespace nomas
