// gather.cu -- temporal_context gather: packs selected archive frames into a contiguous
// INT8 history (comfyui-wiki news, section "单张 4090 配置": the GPU history is limited to
// 18 temporal_context-sampled latent frames).
//
// Packed token j of head h copies archive row (h, src(j)) with
// src(j) = first archive token of the (j / tpf)-th selected frame + j % tpf: 128 code bytes
// of K and of V (4 lanes x 32 bytes each) and the two fp32 scales.  The per-frame source
// offsets travel in the kernel parameters (at most 2048 frames), so the kernel reads
// nothing but the archive.  HBM-bound: 2 x (2 x 128 + 2 x 4) bytes per token and head.
// Each thread copies 32 bytes of a K row and of a V row; the row and frame indices come from
// multiply-shift divisions by host-computed magic numbers.
#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr int kMaxFrames = NOMAS_MAX_GATHER_FRAMES;

struct GatherFrames {
    int32_t src[kMaxFrames];  // first archive token of each selected frame
};

__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherFrames frames, int32_t n_tok,
                                                     int32_t tpf, int32_t heads, FastDiv div_ntok, FastDiv div_tpf,
                                                     const uint4 *__restrict__ ak, const uint4 *__restrict__ av,
                                                     const float *__restrict__ aks, const float *__restrict__ avs,
                                                     int64_t acap, uint4 *__restrict__ dk, uint4 *__restrict__ dv,
                                                     float *__restrict__ dks, float *__restrict__ dvs, int64_t dcap,
                                                     int32_t *__restrict__ index_map) {
    // thread -> (head, packed token, 32-byte quarter of the 128-byte row); head-major so
    // consecutive threads copy consecutive rows of one head (contiguous on both sides within
    // a frame)
    const int64_t total = static_cast<int64_t>(heads) * n_tok * 4;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i & 3);
        const uint32_t r = static_cast<uint32_t>(i >> 2);
        const uint32_t h = fdiv(r, div_ntok);
        const uint32_t j = r - h * static_cast<uint32_t>(n_tok);
        const uint32_t f = fdiv(j, div_tpf);
        const int64_t src = static_cast<int64_t>(frames.src[f]) + (j - f * static_cast<uint32_t>(tpf));
        const int64_t srow = static_cast<int64_t>(h) * acap + src;
        const int64_t drow = static_cast<int64_t>(h) * dcap + j;
        const uint4 k0 = ak[srow * 8 + 2 * c], k1 = ak[srow * 8 + 2 * c + 1];
        const uint4 v0 = av[srow * 8 + 2 * c], v1 = av[srow * 8 + 2 * c + 1];
        dk[drow * 8 + 2 * c] = k0;
        dk[drow * 8 + 2 * c + 1] = k1;
        dv[drow * 8 + 2 * c] = v0;
        dv[drow * 8 + 2 * c + 1] = v1;
        if (c == 0) {
            dks[drow] = aks[srow];
            dvs[drow] = avs[srow];
            if (h == 0 && index_map != nullptr) index_map[j] = static_cast<int32_t>(src);
        }
    }
}

// index_map[j] = archive token of packed token j (for the host-archive gather, whose rows the
// copy engines move)
__global__ void __launch_bounds__(256) index_map_kernel(const __grid_constant__ GatherFrames frames, int32_t n_tok,
                                                        int32_t tpf, FastDiv div_tpf, int32_t *__restrict__ index_map) {
    for (int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; j < n_tok;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint32_t f = fdiv(static_cast<uint32_t>(j), div_tpf);
        index_map[j] = frames.src[f] + static_cast<int32_t>(j - f * static_cast<uint32_t>(tpf));
    }
}

}  // namespace

cudaError_t launch_index_map(const int32_t *src_frame_token, int32_t n_frames, int32_t tpf, int32_t *index_map,
                             cudaStream_t stream) {
    GatherFrames fr;
    for (int i = 0; i < n_frames; ++i) fr.src[i] = src_frame_token[i];
    const int32_t n_tok = n_frames * tpf;
    if (n_tok == 0) return cudaSuccess;
    const int blocks = static_cast<int>((n_tok + 255) / 256 < 1024 ? (n_tok + 255) / 256 : 1024);
    index_map_kernel<<<blocks, 256, 0, stream>>>(fr, n_tok, tpf, make_fastdiv(static_cast<uint32_t>(tpf)), index_map);
    return cudaGetLastError();
}

cudaError_t launch_gather(const nomas_kv_cache &src, const int32_t *src_frame_token, int32_t n_frames,
                          int32_t tpf, nomas_kv_cache &dst, int32_t *index_map, cudaStream_t stream) {
    GatherFrames fr;
    for (int i = 0; i < n_frames; ++i) fr.src[i] = src_frame_token[i];
    const int32_t n_tok = n_frames * tpf;
    const int64_t threads = static_cast<int64_t>(src.heads) * n_tok * 4;
    if (threads == 0) return cudaSuccess;
    int64_t blocks = (threads + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8 * 4;
    if (blocks > cap) blocks = cap;
    gather_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        fr, n_tok, tpf, src.heads, make_fastdiv(static_cast<uint32_t>(n_tok)), make_fastdiv(static_cast<uint32_t>(tpf)),
        reinterpret_cast<const uint4 *>(src.k), reinterpret_cast<const uint4 *>(src.v), src.k_scale, src.v_scale,
        src.capacity, reinterpret_cast<uint4 *>(dst.k), reinterpret_cast<uint4 *>(dst.v), dst.k_scale, dst.v_scale,
        dst.capacity, index_map);
    return cudaGetLastError();
}

}  // namespace nomas
