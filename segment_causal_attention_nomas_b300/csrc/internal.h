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
    const int32_t *seg_off;  // host, n_seg + 1
    const nomas_kv_cache *hist;  // may be null
    int64_t lh;
    float softmax_scale;
    void *out;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    int32_t n_splits;
    int32_t fault;
};
int32_t attn_num_splits(int64_t lq, int64_t lh, int32_t heads, int num_sms);
// The attention workspace, in this order: staged FP16 Q, K, V ([heads][lq][128] each), staged
// FP16 history K, V ([heads][lh][128] each), then the split-KV partials (fp32 O, then LSE).
struct AttnWorkspace {
    size_t cur_bytes, hist_bytes, part_bytes, total;
};
AttnWorkspace attn_workspace_layout(int64_t lq, int64_t lh, int32_t heads, int32_t n_splits);
nomas_status launch_seg_attn(const AttnLaunch &a, cudaStream_t stream, char *err, size_t err_len);

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
