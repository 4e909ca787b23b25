// seg_attn_noalloc.cu -- nomas_seg_attn_noalloc: segment-causal attention whose split-KV
// scratch lives in a fixed device array inside the library, so the caller allocates nothing.
//
// Some callers cannot call cudaMalloc at the point where they run attention: a serving
// process whose framework allocator has already reserved the device memory, or a
// latency-critical loop where cudaMalloc/cudaFree would synchronise the device and stall it.
// They still own and pass the inputs and outputs; only the attention's scratch (the staged FP16
// operands, and the fp32 partial outputs and log-sum-exps that combine_kernel merges when the
// key range is split) comes from here.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes, held by every GPU that
// loads the library until the process exits.  Host code cannot pass the array's name to a
// kernel: on the host that name is a stand-in object, not a device address.  So, once per
// device and with that device current, cudaGetSymbolAddress turns it into the device pointer
// that is handed to the kernels.  The first call on a device does this set-up.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nomas {
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(NOMAS_NOALLOC_SCRATCH_BYTES);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device (nullptr and a message on failure).
void *scratch_address(char *err, size_t err_len) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(err, err_len, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (dev < 0 || dev >= 64) {
        snprintf(err, err_len, "device ordinal %d not supported (0..63)", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            snprintf(err, err_len, "cudaGetSymbolAddress(scratch) on device %d: %s", dev, cudaGetErrorString(e));
            return nullptr;
        }
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace nomas

using namespace nomas;

extern "C" {

nomas_status nomas_seg_attn_noalloc(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16,
                                    int64_t row_stride, int32_t heads, const int32_t *q_seg_offsets, int32_t n_seg,
                                    const nomas_kv_cache *history, float softmax_scale, void *out_bf16, float *lse,
                                    cudaStream_t stream) {
    // the arguments are checked exactly as nomas_seg_attn checks them, before the size check,
    // so a malformed call gets the same status and message as it would there
    SegAttnArgs a{"seg_attn_noalloc", q_bf16, k_cur_bf16, v_cur_bf16, row_stride, heads, q_seg_offsets, n_seg,
                  history, nullptr, softmax_scale, out_bf16, lse, stream};
    int32_t lq;
    int64_t lh;
    nomas_status st = seg_attn_check(a, &lq, &lh);
    if (st != NOMAS_OK) return st;
    if (lq == 0) return seg_attn_run(a, 0, 0, nullptr, 0);
    char msg[320];
    const size_t need = nomas_seg_attn_workspace_size(lq, lh, heads);
    if (need > kNoAllocScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "seg_attn_noalloc: Lq %lld, Lh %lld, %d heads need %zu bytes of scratch; the "
                 "library's fixed scratch holds %zu (use nomas_seg_attn with a caller workspace)",
                 static_cast<long long>(lq), static_cast<long long>(lh), heads, need, kNoAllocScratchBytes);
        set_last_error(msg);
        return NOMAS_ECAPACITY;
    }
    // set-up on the first call on each device: the scratch array's device address
    void *scratch = scratch_address(msg, sizeof(msg));
    if (!scratch) {
        set_last_error(msg);
        return NOMAS_ECUDA;
    }
    // every staged operand, partial and exponent is written by this call before it is read, and
    // the per-head maxima are reset by the call itself, so the previous call's contents never
    // need clearing
    return seg_attn_run(a, lq, lh, scratch, kNoAllocScratchBytes);
}

}  // extern "C"
