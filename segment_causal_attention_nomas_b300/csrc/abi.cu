// abi.cu -- the extern "C" boundary of libnomas (declared in include/nomas.h).
//
// Every entry point validates its arguments on the host before anything is enqueued (on
// error nothing is written or launched and nomas_last_error() says why), then launches the
// kernels of rope_append.cu, gather.cu or seg_attn.cu on the caller's stream.  No entry
// point allocates device memory except nomas_rope_tables_create (its tables, once) and the
// lazily created per-device status word.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "common.cuh"
#include "internal.h"

#define NOMAS_VERSION_STRING "nomas-b300 0.1.0 (sm_103a)"

namespace nomas {

// Library status word: [0] = first failure code since the last check, [1] = where.
__device__ int g_status[2];

namespace {

thread_local char t_err[512] = "";
std::mutex g_mu;
int *g_status_ptr[64] = {nullptr};
int g_sm_count[64] = {0};
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;
int g_fault = 0;  // test hook armed by nomas_debug_inject
int g_attn_variant = 0;  // test hook set by nomas_debug_attn_variant

nomas_status fail(nomas_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return st;
}

nomas_status ok() {
    t_err[0] = '\0';
    return NOMAS_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return (d >= 0 && d < 64) ? d : 0;
}

nomas_status check_segment(const nomas_segment *seg, const char *what) {
    if (!seg) return fail(NOMAS_EINVAL, "%s: segment is NULL", what);
    if (seg->T < 0 || seg->grid_h < 0 || seg->grid_w < 0 || seg->n_text < 0 || seg->t0 < 0)
        return fail(NOMAS_EINVAL, "%s: negative segment field", what);
    const int64_t nv = static_cast<int64_t>(seg->T) * seg->grid_h * seg->grid_w;
    if (nv + seg->n_text > (1ll << 30)) return fail(NOMAS_EUNSUPPORTED, "%s: segment too long", what);
    return NOMAS_OK;
}

SegDesc make_desc(const nomas_segment &s) {
    SegDesc d;
    d.t0 = s.t0;
    d.T = s.T;
    d.gh = s.grid_h;
    d.gw = s.grid_w;
    d.n_text = s.n_text;
    d.n_video = s.T * s.grid_h * s.grid_w;
    d.n_tokens = d.n_video + s.n_text;
    return d;
}

nomas_status check_positions(const nomas_segment &s, const RopeTablesImpl *t, const char *what) {
    const int64_t nv = static_cast<int64_t>(s.T) * s.grid_h * s.grid_w;
    if (nv == 0) return NOMAS_OK;
    // in 64 bits: t0 + T can pass the int32 range, and the kernels index the tables with t0 + t
    const int64_t t_end = static_cast<int64_t>(s.t0) + s.T;
    if (t_end > t->max_pos[0] || s.grid_h > t->max_pos[1] || s.grid_w > t->max_pos[2])
        return fail(NOMAS_EINVAL, "%s: positions (t < %lld, h < %d, w < %d) exceed the RoPE tables (%d, %d, %d)",
                    what, static_cast<long long>(t_end), s.grid_h, s.grid_w, t->max_pos[0], t->max_pos[1],
                    t->max_pos[2]);
    return NOMAS_OK;
}

RopeDev rope_dev(const RopeTablesImpl *t) {
    RopeDev r;
    for (int a = 0; a < 3; ++a) {
        r.cos[a] = t->d_cos[a];
        r.sin[a] = t->d_sin[a];
        r.max_pos[a] = t->max_pos[a];
    }
    return r;
}

nomas_status check_cache(const nomas_kv_cache *c, const char *what) {
    if (!c) return fail(NOMAS_EINVAL, "%s: cache is NULL", what);
    if (c->head_dim != kHeadDim) return fail(NOMAS_EUNSUPPORTED, "%s: head_dim %d (only 128)", what, c->head_dim);
    if (c->heads <= 0) return fail(NOMAS_EINVAL, "%s: heads %d", what, c->heads);
    if (c->capacity < 0 || c->length < 0 || c->length > c->capacity)
        return fail(NOMAS_EINVAL, "%s: length %lld / capacity %lld", what, static_cast<long long>(c->length),
                    static_cast<long long>(c->capacity));
    if (c->capacity % 4 != 0) return fail(NOMAS_EINVAL, "%s: capacity must be a multiple of 4", what);
    if (c->capacity > 0) {
        if (!c->k || !c->v || !c->k_scale || !c->v_scale) return fail(NOMAS_EINVAL, "%s: NULL buffer", what);
        if (!aligned16(c->k) || !aligned16(c->v) || !aligned16(c->k_scale) || !aligned16(c->v_scale))
            return fail(NOMAS_EINVAL, "%s: buffers must be 16-byte aligned", what);
    }
    if (static_cast<int64_t>(c->heads) * c->capacity >= (1ll << 31))
        return fail(NOMAS_EUNSUPPORTED, "%s: heads * capacity must stay below 2^31", what);
    return NOMAS_OK;
}

}  // namespace

void set_last_error(const char *msg) { snprintf(t_err, sizeof(t_err), "%s", msg ? msg : ""); }

int *device_status_word() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[d]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) == cudaSuccess) g_status_ptr[d] = static_cast<int *>(ptr);
    }
    return g_status_ptr[d];
}

int device_sm_count() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
        g_sm_count[d] = n;
    }
    return g_sm_count[d];
}

EncodeTiledFn encode_tiled_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
        g_encode_tried = true;
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

}  // namespace nomas

using namespace nomas;

extern "C" {

const char *nomas_version(void) { return NOMAS_VERSION_STRING; }

const char *nomas_last_error(void) { return t_err; }

const char *nomas_status_string(nomas_status s) {
    switch (s) {
        case NOMAS_OK: return "NOMAS_OK";
        case NOMAS_EINVAL: return "NOMAS_EINVAL: invalid argument";
        case NOMAS_ECAPACITY: return "NOMAS_ECAPACITY: cache capacity exceeded";
        case NOMAS_EUNSUPPORTED: return "NOMAS_EUNSUPPORTED: unsupported configuration";
        case NOMAS_ECUDA: return "NOMAS_ECUDA: CUDA error";
        case NOMAS_ETIMEOUT: return "NOMAS_ETIMEOUT: a kernel's bounded wait gave up";
        case NOMAS_ERANGE: return "NOMAS_ERANGE: input magnitudes beyond the computation's range";
    }
    return "unknown nomas_status";
}

nomas_status nomas_rope_tables_create(float theta, const int32_t split[3], int32_t max_t, int32_t max_h,
                                      int32_t max_w, nomas_rope_tables **out) {
    if (!out || !split) return fail(NOMAS_EINVAL, "rope_tables_create: NULL argument");
    *out = nullptr;
    if (!(theta > 1.0f) || !std::isfinite(theta)) return fail(NOMAS_EINVAL, "rope_tables_create: theta must be > 1");
    if (split[0] + split[1] + split[2] != kHeadDim)
        return fail(NOMAS_EUNSUPPORTED, "rope_tables_create: split must sum to 128");
    // the kernels hand each thread 8 channels inside one axis chunk
    if (split[0] != 16 || split[1] != 56 || split[2] != 56)
        return fail(NOMAS_EUNSUPPORTED, "rope_tables_create: only the [16, 56, 56] split is built");
    if (max_t <= 0 || max_h <= 0 || max_w <= 0 || max_t > (1 << 20) || max_h > (1 << 20) || max_w > (1 << 20))
        return fail(NOMAS_EINVAL, "rope_tables_create: table sizes must be in [1, 2^20]");
    RopeTablesImpl *t = new (std::nothrow) RopeTablesImpl;
    if (!t) return fail(NOMAS_ECUDA, "rope_tables_create: out of host memory");
    memset(t, 0, sizeof(*t));
    t->device = current_device();
    const int32_t maxp[3] = {max_t, max_h, max_w};
    for (int a = 0; a < 3; ++a) {
        t->split[a] = split[a];
        t->max_pos[a] = maxp[a];
        const int half = split[a] / 2;
        const size_t n = static_cast<size_t>(maxp[a]) * half;
        t->h_cos[a] = static_cast<float *>(malloc(n * sizeof(float)));
        t->h_sin[a] = static_cast<float *>(malloc(n * sizeof(float)));
        if (!t->h_cos[a] || !t->h_sin[a]) {
            nomas_rope_tables_destroy(reinterpret_cast<nomas_rope_tables *>(t));
            return fail(NOMAS_ECUDA, "rope_tables_create: out of host memory");
        }
        // angle of pair i at position p: p * theta^(-2i/d), evaluated in double, rounded once
        for (int32_t pos = 0; pos < maxp[a]; ++pos)
            for (int i = 0; i < half; ++i) {
                const double omega = std::pow(static_cast<double>(theta), -2.0 * static_cast<double>(i) /
                                                                              static_cast<double>(split[a]));
                const double ang = static_cast<double>(pos) * omega;
                t->h_cos[a][static_cast<size_t>(pos) * half + i] = static_cast<float>(std::cos(ang));
                t->h_sin[a][static_cast<size_t>(pos) * half + i] = static_cast<float>(std::sin(ang));
            }
        const bool dev_ok =
            cudaMalloc(&t->d_cos[a], n * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&t->d_sin[a], n * sizeof(float)) == cudaSuccess &&
            cudaMemcpy(t->d_cos[a], t->h_cos[a], n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(t->d_sin[a], t->h_sin[a], n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess;
        if (!dev_ok) {
            cudaGetLastError();
            nomas_rope_tables_destroy(reinterpret_cast<nomas_rope_tables *>(t));
            return fail(NOMAS_ECUDA, "rope_tables_create: device allocation/copy failed");
        }
    }
    *out = reinterpret_cast<nomas_rope_tables *>(t);
    return ok();
}

void nomas_rope_tables_destroy(nomas_rope_tables *tables) {
    RopeTablesImpl *t = reinterpret_cast<RopeTablesImpl *>(tables);
    if (!t) return;
    for (int a = 0; a < 3; ++a) {
        if (t->d_cos[a]) cudaFree(t->d_cos[a]);
        if (t->d_sin[a]) cudaFree(t->d_sin[a]);
        free(t->h_cos[a]);
        free(t->h_sin[a]);
    }
    delete t;
}

nomas_status nomas_rope_tables_read(const nomas_rope_tables *tables, int32_t axis, float *cos_out, float *sin_out) {
    const RopeTablesImpl *t = reinterpret_cast<const RopeTablesImpl *>(tables);
    if (!t || !cos_out || !sin_out) return fail(NOMAS_EINVAL, "rope_tables_read: NULL argument");
    if (axis < 0 || axis > 2) return fail(NOMAS_EINVAL, "rope_tables_read: axis must be 0, 1 or 2");
    const size_t n = static_cast<size_t>(t->max_pos[axis]) * (t->split[axis] / 2);
    memcpy(cos_out, t->h_cos[axis], n * sizeof(float));
    memcpy(sin_out, t->h_sin[axis], n * sizeof(float));
    return ok();
}

nomas_status nomas_rope3d(const void *x_bf16, void *y_bf16, int64_t row_stride, const nomas_segment *seg,
                          int32_t heads, const nomas_rope_tables *tables, cudaStream_t stream) {
    nomas_status st = check_segment(seg, "rope3d");
    if (st != NOMAS_OK) return st;
    const RopeTablesImpl *t = reinterpret_cast<const RopeTablesImpl *>(tables);
    if (!t) return fail(NOMAS_EINVAL, "rope3d: tables is NULL");
    if (heads <= 0) return fail(NOMAS_EINVAL, "rope3d: heads %d", heads);
    if (row_stride < static_cast<int64_t>(heads) * kHeadDim || row_stride % 8 != 0)
        return fail(NOMAS_EINVAL, "rope3d: row_stride %lld (>= heads*128, multiple of 8)",
                    static_cast<long long>(row_stride));
    const SegDesc d = make_desc(*seg);
    if (d.n_tokens == 0) return ok();
    if (static_cast<int64_t>(d.n_tokens) * heads >= (1ll << 31))
        return fail(NOMAS_EUNSUPPORTED, "rope3d: tokens * heads must stay below 2^31");
    if (!x_bf16 || !y_bf16 || !aligned16(x_bf16) || !aligned16(y_bf16))
        return fail(NOMAS_EINVAL, "rope3d: x/y must be non-NULL and 16-byte aligned");
    if ((st = check_positions(*seg, t, "rope3d")) != NOMAS_OK) return st;
    if (x_bf16 != y_bf16) {
        const char *xb = static_cast<const char *>(x_bf16), *yb = static_cast<const char *>(y_bf16);
        const int64_t span =
            (static_cast<int64_t>(d.n_tokens - 1) * row_stride + static_cast<int64_t>(heads) * kHeadDim) * 2;
        if (xb < yb + span && yb < xb + span) return fail(NOMAS_EINVAL, "rope3d: x and y overlap (and differ)");
    }
    cudaError_t e = launch_rope3d(x_bf16, y_bf16, row_stride, d, heads, rope_dev(t), stream);
    if (e != cudaSuccess) return fail(NOMAS_ECUDA, "rope3d launch: %s", cudaGetErrorString(e));
    return ok();
}

nomas_status nomas_kv_append_quant(nomas_kv_cache *cache, const void *k_bf16, const void *v_bf16,
                                   int64_t row_stride, const nomas_segment *seg, const nomas_rope_tables *tables,
                                   cudaStream_t stream) {
    nomas_status st = check_cache(cache, "kv_append_quant");
    if (st != NOMAS_OK) return st;
    if ((st = check_segment(seg, "kv_append_quant")) != NOMAS_OK) return st;
    const SegDesc d = make_desc(*seg);
    if (cache->length + d.n_tokens > cache->capacity)
        return fail(NOMAS_ECAPACITY, "kv_append_quant: length %lld + %d tokens > capacity %lld",
                    static_cast<long long>(cache->length), d.n_tokens, static_cast<long long>(cache->capacity));
    const RopeTablesImpl *t = reinterpret_cast<const RopeTablesImpl *>(tables);
    if (!t) return fail(NOMAS_EINVAL, "kv_append_quant: tables is NULL");
    if (d.n_tokens == 0) return ok();
    if (row_stride < static_cast<int64_t>(cache->heads) * kHeadDim || row_stride % 8 != 0)
        return fail(NOMAS_EINVAL, "kv_append_quant: row_stride %lld", static_cast<long long>(row_stride));
    if (!k_bf16 || !v_bf16 || !aligned16(k_bf16) || !aligned16(v_bf16))
        return fail(NOMAS_EINVAL, "kv_append_quant: k/v must be non-NULL and 16-byte aligned");
    if ((st = check_positions(*seg, t, "kv_append_quant")) != NOMAS_OK) return st;
    cudaError_t e = launch_append_quant(k_bf16, v_bf16, row_stride, d, cache->heads, rope_dev(t), cache->k, cache->v,
                                        cache->k_scale, cache->v_scale, cache->capacity, cache->length, stream);
    if (e != cudaSuccess) return fail(NOMAS_ECUDA, "kv_append_quant launch: %s", cudaGetErrorString(e));
    cache->length += d.n_tokens;
    return ok();
}

}  // extern "C"

namespace {

// Checks shared by both gather entry points; fills src_tok with each frame's first archive token.
nomas_status check_gather(const char *what, const nomas_kv_cache *archive, const int32_t *frame_token_offset,
                          int32_t n_archive_frames, int32_t tokens_per_frame, const int32_t *frames,
                          int32_t n_frames, const nomas_kv_cache *dst, const int32_t *index_map, int32_t *src_tok) {
    nomas_status st = check_cache(archive, what);
    if (st != NOMAS_OK) return st;
    if ((st = check_cache(dst, what)) != NOMAS_OK) return st;
    if (archive->heads != dst->heads) return fail(NOMAS_EINVAL, "%s: heads differ", what);
    if (n_frames < 0 || tokens_per_frame <= 0 || n_archive_frames < 0)
        return fail(NOMAS_EINVAL, "%s: negative count", what);
    if (n_frames > NOMAS_MAX_GATHER_FRAMES)
        return fail(NOMAS_EUNSUPPORTED, "%s: %d frames (max %d)", what, n_frames, NOMAS_MAX_GATHER_FRAMES);
    if (n_frames > 0 && (!frames || !frame_token_offset)) return fail(NOMAS_EINVAL, "%s: NULL frame list", what);
    const int64_t n = static_cast<int64_t>(n_frames) * tokens_per_frame;
    if (n > dst->capacity)
        return fail(NOMAS_ECAPACITY, "%s: %lld tokens > dst capacity %lld", what, static_cast<long long>(n),
                    static_cast<long long>(dst->capacity));
    if (index_map && !aligned16(index_map)) return fail(NOMAS_EINVAL, "%s: index_map misaligned", what);
    for (int i = 0; i < n_frames; ++i) {
        if (frames[i] < 0 || frames[i] >= n_archive_frames)
            return fail(NOMAS_EINVAL, "%s: frame %d out of range", what, frames[i]);
        if (i > 0 && frames[i] <= frames[i - 1])
            return fail(NOMAS_EINVAL, "%s: frames must be strictly increasing", what);
        const int64_t s = frame_token_offset[frames[i]];
        if (s < 0 || s + tokens_per_frame > archive->length)
            return fail(NOMAS_EINVAL, "%s: frame %d tokens [%lld, %lld) outside archive length %lld", what, frames[i],
                        static_cast<long long>(s), static_cast<long long>(s + tokens_per_frame),
                        static_cast<long long>(archive->length));
        src_tok[i] = static_cast<int32_t>(s);
    }
    if (archive->k == dst->k) return fail(NOMAS_EINVAL, "%s: dst aliases the archive", what);
    return NOMAS_OK;
}

// The sizes nomas_seg_attn accepts (its checks refuse larger Lq, Lh or head counts), so the
// workspace formulas never see a product that wraps.
bool attn_size_supported(int64_t lq, int64_t lh, int32_t heads) {
    return lq > 0 && lq < (1 << 30) && lh >= 0 && lh < (1 << 30) && heads > 0 && heads <= NOMAS_MAX_ATTN_HEADS &&
           2ll * heads * lh < (1ll << 31);
}

bool is_pinned_host(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of a failed query
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

nomas_status nomas_kv_gather_context(const nomas_kv_cache *archive, const int32_t *frame_token_offset,
                                     int32_t n_archive_frames, int32_t tokens_per_frame, const int32_t *frames,
                                     int32_t n_frames, nomas_kv_cache *dst, int32_t *index_map,
                                     cudaStream_t stream) {
    static thread_local int32_t src_tok[NOMAS_MAX_GATHER_FRAMES];
    nomas_status st = check_gather("kv_gather_context", archive, frame_token_offset, n_archive_frames,
                                   tokens_per_frame, frames, n_frames, dst, index_map, src_tok);
    if (st != NOMAS_OK) return st;
    const int64_t n = static_cast<int64_t>(n_frames) * tokens_per_frame;
    if (n > 0) {
        cudaError_t e = launch_gather(*archive, src_tok, n_frames, tokens_per_frame, *dst, index_map, stream);
        if (e != cudaSuccess) return fail(NOMAS_ECUDA, "kv_gather_context launch: %s", cudaGetErrorString(e));
    }
    dst->length = n;
    return ok();
}

nomas_status nomas_kv_gather_context_host(const nomas_kv_cache *archive, const int32_t *frame_token_offset,
                                          int32_t n_archive_frames, int32_t tokens_per_frame, const int32_t *frames,
                                          int32_t n_frames, nomas_kv_cache *dst, int32_t *index_map,
                                          cudaStream_t stream) {
    static thread_local int32_t src_tok[NOMAS_MAX_GATHER_FRAMES];
    nomas_status st = check_gather("kv_gather_context_host", archive, frame_token_offset, n_archive_frames,
                                   tokens_per_frame, frames, n_frames, dst, index_map, src_tok);
    if (st != NOMAS_OK) return st;
    if (archive->capacity > 0 && (!is_pinned_host(archive->k) || !is_pinned_host(archive->v) ||
                                  !is_pinned_host(archive->k_scale) || !is_pinned_host(archive->v_scale)))
        return fail(NOMAS_EINVAL, "kv_gather_context_host: archive buffers must be pinned host memory");
    const int64_t n = static_cast<int64_t>(n_frames) * tokens_per_frame;
    const int64_t h = archive->heads, acap = archive->capacity, dcap = dst->capacity;
    // one 2-D copy per run of frames consecutive in the archive, per array, all heads at once
    for (int i = 0; i < n_frames;) {
        int r = i + 1;
        while (r < n_frames && src_tok[r] == src_tok[r - 1] + tokens_per_frame) ++r;
        const int64_t s = src_tok[i], d = static_cast<int64_t>(i) * tokens_per_frame;
        const int64_t rows = static_cast<int64_t>(r - i) * tokens_per_frame;
        struct Part {
            const void *src;
            void *dst;
            size_t elem;
        } parts[4] = {{archive->k, dst->k, kHeadDim},
                      {archive->v, dst->v, kHeadDim},
                      {archive->k_scale, dst->k_scale, sizeof(float)},
                      {archive->v_scale, dst->v_scale, sizeof(float)}};
        for (const Part &pt : parts) {
            cudaError_t e = cudaMemcpy2DAsync(static_cast<char *>(pt.dst) + d * pt.elem, dcap * pt.elem,
                                              static_cast<const char *>(pt.src) + s * pt.elem, acap * pt.elem,
                                              rows * pt.elem, h, cudaMemcpyHostToDevice, stream);
            if (e != cudaSuccess) return fail(NOMAS_ECUDA, "kv_gather_context_host copy: %s", cudaGetErrorString(e));
        }
        i = r;
    }
    if (index_map && n > 0) {
        cudaError_t e = launch_index_map(src_tok, n_frames, tokens_per_frame, index_map, stream);
        if (e != cudaSuccess) return fail(NOMAS_ECUDA, "kv_gather_context_host index map: %s", cudaGetErrorString(e));
    }
    dst->length = n;
    return ok();
}

size_t nomas_qkv_project_workspace_size(int32_t heads, int32_t hidden) {
    if (heads <= 0 || hidden <= 0) return 0;
    return qkv_project_workspace_bytes(heads, hidden);
}

}  // extern "C"

namespace {

nomas_status qkv_project(const char *what, const void *x_bf16, int64_t x_row_stride, int32_t hidden,
                         const int8_t *w_codes, const float *w_scale, int32_t heads, const nomas_segment *seg,
                         const nomas_rope_tables *tables, void *qkv_bf16, int64_t out_row_stride, void *workspace,
                         size_t workspace_bytes, nomas_kv_cache *cache, cudaStream_t stream) {
    nomas_status st = check_segment(seg, what);
    if (st != NOMAS_OK) return st;
    const RopeTablesImpl *t = reinterpret_cast<const RopeTablesImpl *>(tables);
    if (!t) return fail(NOMAS_EINVAL, "%s: tables is NULL", what);
    if (heads <= 0 || heads % 2 != 0 || heads > NOMAS_MAX_ATTN_HEADS)
        return fail(NOMAS_EUNSUPPORTED, "%s: heads %d (even, 2..%d)", what, heads, NOMAS_MAX_ATTN_HEADS);
    if (hidden < 64 || hidden % 64 != 0 || hidden > 65536)
        return fail(NOMAS_EUNSUPPORTED, "%s: hidden %d (a multiple of 64, at most 65536)", what, hidden);
    const int64_t n_out = 3ll * heads * kHeadDim;
    if (x_row_stride < hidden || x_row_stride % 8 != 0)
        return fail(NOMAS_EINVAL, "%s: x_row_stride %lld", what, static_cast<long long>(x_row_stride));
    if (out_row_stride < n_out || out_row_stride % 8 != 0)
        return fail(NOMAS_EINVAL, "%s: out_row_stride %lld", what, static_cast<long long>(out_row_stride));
    const SegDesc d = make_desc(*seg);
    if (cache) {
        if ((st = check_cache(cache, what)) != NOMAS_OK) return st;
        if (cache->heads != heads) return fail(NOMAS_EINVAL, "%s: cache has %d heads, not %d", what, cache->heads, heads);
        if (cache->length + d.n_tokens > cache->capacity)
            return fail(NOMAS_ECAPACITY, "%s: length %lld + %d tokens > capacity %lld", what,
                        static_cast<long long>(cache->length), d.n_tokens, static_cast<long long>(cache->capacity));
    }
    if (d.n_tokens == 0) return ok();
    if (!x_bf16 || !w_codes || !w_scale || !qkv_bf16 || !aligned16(x_bf16) || !aligned16(w_codes) ||
        !aligned16(w_scale) || !aligned16(qkv_bf16))
        return fail(NOMAS_EINVAL, "%s: device buffers must be non-NULL and 16-byte aligned", what);
    if ((st = check_positions(*seg, t, what)) != NOMAS_OK) return st;
    const size_t need = qkv_project_workspace_bytes(heads, hidden);
    if (workspace_bytes < need || !workspace || !aligned16(workspace))
        return fail(NOMAS_EINVAL, "%s: workspace needs %zu bytes (16-byte aligned), got %zu", what, need,
                    workspace_bytes);
    QkvLaunch a;
    a.x = x_bf16;
    a.x_row_stride = x_row_stride;
    a.hidden = hidden;
    a.heads = heads;
    a.lq = d.n_tokens;
    a.w_codes = w_codes;
    a.w_scale = w_scale;
    a.seg = d;
    a.rope = rope_dev(t);
    a.out = qkv_bf16;
    a.out_row_stride = out_row_stride;
    a.workspace = workspace;
    a.cache = cache;
    if (!device_status_word()) return fail(NOMAS_ECUDA, "%s: status word unavailable", what);
    char err[256] = "";
    st = launch_qkv_project(a, stream, err, sizeof(err));
    if (st != NOMAS_OK) return fail(st, "%s: %s", what, err);
    if (cache) cache->length += d.n_tokens;
    return ok();
}

}  // namespace

extern "C" {

nomas_status nomas_qkv_project_rope(const void *x_bf16, int64_t x_row_stride, int32_t hidden, const int8_t *w_codes,
                                    const float *w_scale, int32_t heads, const nomas_segment *seg,
                                    const nomas_rope_tables *tables, void *qkv_bf16, int64_t out_row_stride,
                                    void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return qkv_project("qkv_project_rope", x_bf16, x_row_stride, hidden, w_codes, w_scale, heads, seg, tables,
                       qkv_bf16, out_row_stride, workspace, workspace_bytes, nullptr, stream);
}

nomas_status nomas_qkv_project_rope_append(const void *x_bf16, int64_t x_row_stride, int32_t hidden,
                                           const int8_t *w_codes, const float *w_scale, int32_t heads,
                                           const nomas_segment *seg, const nomas_rope_tables *tables, void *qkv_bf16,
                                           int64_t out_row_stride, void *workspace, size_t workspace_bytes,
                                           nomas_kv_cache *cache, cudaStream_t stream) {
    if (!cache) return fail(NOMAS_EINVAL, "qkv_project_rope_append: cache is NULL");
    return qkv_project("qkv_project_rope_append", x_bf16, x_row_stride, hidden, w_codes, w_scale, heads, seg, tables,
                       qkv_bf16, out_row_stride, workspace, workspace_bytes, cache, stream);
}

nomas_status nomas_camera_tokens(const float *c2w, int32_t n_frames, float translation_scale, float rotation_scale,
                                 float *tokens, cudaStream_t stream) {
    if (n_frames <= 0 || n_frames % 4 != 0 || n_frames > (1 << 24))
        return fail(NOMAS_EINVAL, "camera_tokens: n_frames %d (a positive multiple of 4, at most 2^24)", n_frames);
    if (!std::isfinite(translation_scale) || !std::isfinite(rotation_scale))
        return fail(NOMAS_EINVAL, "camera_tokens: scales must be finite");
    if (!c2w || !tokens || !aligned16(c2w) || !aligned16(tokens))
        return fail(NOMAS_EINVAL, "camera_tokens: device buffers must be non-NULL and 16-byte aligned");
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(c2w), a1 = a0 + 64ull * n_frames;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(tokens), b1 = b0 + 64ull * n_frames;
    if (a0 < b1 && b0 < a1) return fail(NOMAS_EINVAL, "camera_tokens: tokens overlaps c2w");
    cudaError_t e = launch_camera_tokens(c2w, n_frames, translation_scale, rotation_scale, tokens, stream);
    if (e != cudaSuccess) return fail(NOMAS_ECUDA, "camera_tokens launch: %s", cudaGetErrorString(e));
    return ok();
}

nomas_status nomas_camera_cross_attn(const void *q_bf16, int64_t q_row_stride, int32_t lq, int32_t heads,
                                     const void *k_cam_bf16, const void *v_cam_bf16, int64_t cam_row_stride,
                                     int32_t n_cam, float softmax_scale, void *out_bf16, int64_t out_row_stride,
                                     cudaStream_t stream) {
    if (heads <= 0 || lq < 0 || n_cam < 1)
        return fail(NOMAS_EINVAL, "camera_cross_attn: heads %d, lq %d, n_cam %d", heads, lq, n_cam);
    if (heads > NOMAS_MAX_ATTN_HEADS)
        return fail(NOMAS_EUNSUPPORTED, "camera_cross_attn: %d heads (max %d)", heads, NOMAS_MAX_ATTN_HEADS);
    if (n_cam > NOMAS_MAX_CAMERA_TOKENS)
        return fail(NOMAS_EUNSUPPORTED, "camera_cross_attn: %d camera tokens (max %d)", n_cam,
                    NOMAS_MAX_CAMERA_TOKENS);
    if ((static_cast<int64_t>(lq) + 127) / 128 * heads >= (1ll << 31))
        return fail(NOMAS_EUNSUPPORTED, "camera_cross_attn: %d tokens x %d heads is too many tiles", lq, heads);
    if (!std::isfinite(softmax_scale) || softmax_scale < 0.0f)
        return fail(NOMAS_EINVAL, "camera_cross_attn: softmax_scale must be finite and >= 0");
    const int64_t width = static_cast<int64_t>(heads) * kHeadDim;
    for (int64_t s : {q_row_stride, cam_row_stride, out_row_stride})
        if (s < width || s % 8 != 0)
            return fail(NOMAS_EINVAL, "camera_cross_attn: row stride %lld (a multiple of 8, >= %lld)",
                        static_cast<long long>(s), static_cast<long long>(width));
    if (lq == 0) return ok();
    if (!q_bf16 || !k_cam_bf16 || !v_cam_bf16 || !out_bf16 || !aligned16(q_bf16) || !aligned16(k_cam_bf16) ||
        !aligned16(v_cam_bf16) || !aligned16(out_bf16))
        return fail(NOMAS_EINVAL, "camera_cross_attn: device buffers must be non-NULL and 16-byte aligned");
    if (out_bf16 == q_bf16 && out_row_stride != q_row_stride)
        return fail(NOMAS_EINVAL, "camera_cross_attn: out aliases q with another stride");
    if (!device_status_word()) return fail(NOMAS_ECUDA, "camera_cross_attn: status word unavailable");
    CamLaunch a;
    a.q = q_bf16;
    a.q_row_stride = q_row_stride;
    a.lq = lq;
    a.heads = heads;
    a.k = k_cam_bf16;
    a.v = v_cam_bf16;
    a.cam_row_stride = cam_row_stride;
    a.n_cam = n_cam;
    a.softmax_scale = softmax_scale;
    a.out = out_bf16;
    a.out_row_stride = out_row_stride;
    char err[256] = "";
    nomas_status st = launch_camera_xattn(a, stream, err, sizeof(err));
    if (st != NOMAS_OK) return fail(st, "camera_cross_attn: %s", err);
    return ok();
}

size_t nomas_seg_attn_workspace_size(int64_t lq, int64_t lh, int32_t heads) {
    if (!attn_size_supported(lq, lh, heads)) return 0;
    return attn_workspace_layout(lq, lh, heads, attn_num_splits(lq, lh, heads, device_sm_count()), true).total;
}

size_t nomas_seg_attn_staged_workspace_size(int64_t lq, int64_t lh, int32_t heads) {
    if (!attn_size_supported(lq, lh, heads)) return 0;
    return attn_workspace_layout(lq, lh, heads, attn_num_splits(lq, lh, heads, device_sm_count()), false).total;
}

size_t nomas_staged_history_size(int64_t capacity, int32_t heads) {
    if (capacity <= 0 || heads <= 0) return 0;
    return staged_history_bytes(capacity, heads);
}

}  // extern "C"

namespace nomas {

nomas_status seg_attn_check(const SegAttnArgs &a, int32_t *lq_out, int64_t *lh_out) {
    const char *what = a.what;
    *lq_out = 0;
    *lh_out = 0;
    if (a.heads <= 0) return fail(NOMAS_EINVAL, "%s: heads %d", what, a.heads);
    if (a.heads > NOMAS_MAX_ATTN_HEADS)
        return fail(NOMAS_EUNSUPPORTED, "%s: %d heads (max %d)", what, a.heads, NOMAS_MAX_ATTN_HEADS);
    if (a.n_seg < 1 || !a.offs) return fail(NOMAS_EINVAL, "%s: need n_seg >= 1 and offsets", what);
    if (a.n_seg > NOMAS_MAX_SEGMENTS)
        return fail(NOMAS_EUNSUPPORTED, "%s: %d segments (max %d)", what, a.n_seg, NOMAS_MAX_SEGMENTS);
    if (a.offs[0] != 0) return fail(NOMAS_EINVAL, "%s: offsets[0] must be 0", what);
    for (int s = 0; s < a.n_seg; ++s)
        if (a.offs[s + 1] < a.offs[s]) return fail(NOMAS_EINVAL, "%s: offsets must not decrease", what);
    const int32_t lq = a.offs[a.n_seg];
    if (lq < 0 || lq >= (1 << 30)) return fail(NOMAS_EINVAL, "%s: Lq %d", what, lq);
    if (lq == 0) return NOMAS_OK;
    if (!std::isfinite(a.softmax_scale) || a.softmax_scale < 0.0f)
        return fail(NOMAS_EINVAL, "%s: softmax_scale must be finite and >= 0", what);
    if (a.row_stride < static_cast<int64_t>(a.heads) * kHeadDim || a.row_stride % 8 != 0)
        return fail(NOMAS_EINVAL, "%s: row_stride %lld", what, static_cast<long long>(a.row_stride));
    if (!a.q || !a.k || !a.v || !a.out) return fail(NOMAS_EINVAL, "%s: NULL q/k/v/out", what);
    if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.out) || (a.lse && !aligned16(a.lse)))
        return fail(NOMAS_EINVAL, "%s: device buffers must be 16-byte aligned", what);
    int64_t lh = 0;
    if (a.history) {
        nomas_status st = check_cache(a.history, what);
        if (st != NOMAS_OK) return st;
        if (a.history->heads != a.heads)
            return fail(NOMAS_EINVAL, "%s: history heads %d != %d", what, a.history->heads, a.heads);
        lh = a.history->length;
    } else if (a.staged) {
        const nomas_staged_history *h = a.staged;
        if (h->length < 0 || h->capacity < 0 || h->length > h->capacity)
            return fail(NOMAS_EINVAL, "%s: staged history length %lld / capacity %lld", what,
                        static_cast<long long>(h->length), static_cast<long long>(h->capacity));
        if (h->length > 0) {
            if (h->heads != a.heads)
                return fail(NOMAS_EINVAL, "%s: staged history heads %d != %d", what, h->heads, a.heads);
            if (!h->data || !aligned16(h->data) || h->bytes < staged_history_bytes(h->capacity, h->heads))
                return fail(NOMAS_EINVAL, "%s: staged history buffer (non-NULL, 16-byte aligned, %zu bytes)", what,
                            staged_history_bytes(h->capacity, h->heads));
        }
        lh = h->length;
    }
    if (lh >= (1 << 30) || 2ll * a.heads * lh >= (1ll << 31))
        return fail(NOMAS_EUNSUPPORTED, "%s: history too long (heads x rows must stay below 2^30)", what);
    *lq_out = lq;
    *lh_out = lh;
    return NOMAS_OK;
}

nomas_status seg_attn_run(const SegAttnArgs &a, int32_t lq, int64_t lh, void *workspace, size_t workspace_bytes) {
    const char *what = a.what;
    if (lq == 0) return ok();
    const bool stage_here = a.history != nullptr && lh > 0;
    const int32_t n_splits = attn_num_splits(lq, lh, a.heads, device_sm_count());
    const AttnWorkspace lay = attn_workspace_layout(lq, lh, a.heads, n_splits, stage_here);
    if (workspace_bytes < lay.total || !workspace || !aligned16(workspace))
        return fail(NOMAS_EINVAL, "%s: workspace needs %zu bytes (16-byte aligned), got %zu", what, lay.total,
                    workspace_bytes);
    if (!device_status_word()) return fail(NOMAS_ECUDA, "%s: status word unavailable", what);
    AttnLaunch l;
    memset(&l, 0, sizeof(l));
    l.q = a.q;
    l.k = a.k;
    l.v = a.v;
    l.row_stride = a.row_stride;
    l.heads = a.heads;
    l.lq = lq;
    l.n_seg = a.n_seg;
    l.seg_off = a.offs;
    l.lh = lh;
    l.softmax_scale = a.softmax_scale;
    l.out = a.out;
    l.lse = a.lse;
    l.workspace = workspace;
    l.part_off = lay.part_off;
    l.qexp_off = lay.qexp_off;
    l.max_off = lay.max_off;
    l.n_splits = n_splits;
    char err[256] = "";
    if (stage_here) {
        // the INT8 history is staged into the workspace's history block, then attended
        void *block = static_cast<uint8_t *>(workspace) + lay.hist_off;
        nomas_status st = launch_stage_history(*a.history, lh, block, lh, a.stream, err, sizeof(err));
        if (st != NOMAS_OK) return fail(st, "%s: %s", what, err);
        l.hist_block = block;
        l.hist_cap = lh;
    } else if (a.staged && lh > 0) {
        l.hist_block = a.staged->data;
        l.hist_cap = a.staged->capacity;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        l.fault = g_fault;
        g_fault = 0;
        l.variant = g_attn_variant;
    }
    nomas_status st = launch_seg_attn(l, a.stream, err, sizeof(err));
    if (st != NOMAS_OK) return fail(st, "%s: %s", what, err);
    return ok();
}

}  // namespace nomas

extern "C" {

nomas_status nomas_seg_attn(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16, int64_t row_stride,
                            int32_t heads, const int32_t *q_seg_offsets, int32_t n_seg, const nomas_kv_cache *history,
                            float softmax_scale, void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    SegAttnArgs a{"seg_attn", q_bf16, k_cur_bf16, v_cur_bf16, row_stride, heads, q_seg_offsets, n_seg, history,
                  nullptr, softmax_scale, out_bf16, lse, stream};
    int32_t lq;
    int64_t lh;
    nomas_status st = seg_attn_check(a, &lq, &lh);
    if (st != NOMAS_OK) return st;
    return seg_attn_run(a, lq, lh, workspace, workspace_bytes);
}

nomas_status nomas_seg_attn_stage_history(const nomas_kv_cache *history, nomas_staged_history *staged,
                                          cudaStream_t stream) {
    nomas_status st = check_cache(history, "seg_attn_stage_history");
    if (st != NOMAS_OK) return st;
    if (!staged) return fail(NOMAS_EINVAL, "seg_attn_stage_history: staged is NULL");
    const int64_t lh = history->length;
    if (staged->heads != history->heads)
        return fail(NOMAS_EINVAL, "seg_attn_stage_history: staged heads %d != history heads %d", staged->heads,
                    history->heads);
    if (lh > staged->capacity)
        return fail(NOMAS_ECAPACITY, "seg_attn_stage_history: %lld history rows > staged capacity %lld",
                    static_cast<long long>(lh), static_cast<long long>(staged->capacity));
    if (lh >= (1 << 30) || 2ll * history->heads * lh >= (1ll << 31))
        return fail(NOMAS_EUNSUPPORTED, "seg_attn_stage_history: history too long");
    if (lh > 0 && (!staged->data || !aligned16(staged->data) ||
                   staged->bytes < staged_history_bytes(staged->capacity, staged->heads)))
        return fail(NOMAS_EINVAL, "seg_attn_stage_history: staged buffer (non-NULL, 16-byte aligned, %zu bytes)",
                    staged_history_bytes(staged->capacity, staged->heads));
    if (lh > 0) {
        char err[256] = "";
        st = launch_stage_history(*history, lh, staged->data, staged->capacity, stream, err, sizeof(err));
        if (st != NOMAS_OK) return fail(st, "seg_attn_stage_history: %s", err);
    }
    staged->length = lh;
    return ok();
}

nomas_status nomas_seg_attn_staged(const void *q_bf16, const void *k_cur_bf16, const void *v_cur_bf16,
                                   int64_t row_stride, int32_t heads, const int32_t *q_seg_offsets, int32_t n_seg,
                                   const nomas_staged_history *history, float softmax_scale, void *out_bf16,
                                   float *lse, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    SegAttnArgs a{"seg_attn_staged", q_bf16, k_cur_bf16, v_cur_bf16, row_stride, heads, q_seg_offsets, n_seg,
                  nullptr, history, softmax_scale, out_bf16, lse, stream};
    int32_t lq;
    int64_t lh;
    nomas_status st = seg_attn_check(a, &lq, &lh);
    if (st != NOMAS_OK) return st;
    return seg_attn_run(a, lq, lh, workspace, workspace_bytes);
}

nomas_status nomas_stream_check(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(NOMAS_ECUDA, "stream_check: %s", cudaGetErrorString(e));
    int *w = device_status_word();
    if (!w) return fail(NOMAS_ECUDA, "stream_check: status word unavailable");
    int h[2] = {0, 0};
    e = cudaMemcpy(h, w, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(NOMAS_ECUDA, "stream_check: %s", cudaGetErrorString(e));
    if (h[0] != 0) {
        const int zero[2] = {0, 0};
        cudaMemcpy(w, zero, sizeof(zero), cudaMemcpyHostToDevice);
        return fail(static_cast<nomas_status>(h[0]), "stream_check: device status %d at wait %d", h[0], h[1]);
    }
    return ok();
}

void nomas_debug_inject(int32_t what) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_fault = what;
}

void nomas_debug_attn_variant(int32_t variant) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_attn_variant = variant == 1 || variant == 2 ? variant : 0;
}

}  // extern "C"
