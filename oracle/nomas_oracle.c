/*
 * nomas_oracle.c -- plain, slow CPU oracle for the segment-causal attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm may load this.  It shares no code, header, table or
 * constant generator with the CUDA library: every step is written out from the
 * statement of the method, in float64 wherever the method leaves the precision open.
 *
 * Sources (the Hy-Nomas web pages):
 *   [comfyui]  comfyui-wiki news "Hy-Nomas：腾讯混元交互式世界模型" --
 *              section "一个世界，分段生成" (segments attend to every earlier
 *              segment's K/V cache; attention is causal across segments),
 *              section "模型内部", architecture table (16 heads x 128; 3D RoPE
 *              sizes [16, 56, 56], theta 256; patch 1x1x1),
 *              section "单张 4090 配置" (cached K/V stored INT8, attention computed
 *              in BF16; GPU history limited to 18 temporal_context-sampled frames).
 *   [huawei]   huaweicloud blog, section 2.1 (each segment's text/video K,V cached and
 *              passed to the next segment).
 * The pages print no formula; the rules below are the plainest reading of them,
 * with the quantisation rule of the benchmark spec (symmetric per-token-per-head
 * absmax, fp32 scale = absmax/127, round-half-even, clamp to +-127).
 *
 * Compiled with gcc -O2 -ffp-contract=off (no FMA contraction, IEEE division).
 * Parity pins: see tests/test_oracle_pins.py.  Every function here is pinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- BF16 bits */

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round an fp32 value to the nearest BF16, ties to even (IEEE RNE). */
static uint16_t float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)           /* NaN stays NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

double orc_bf16_to_double(uint16_t b) { return (double)bf16_to_float(b); }
uint16_t orc_float_to_bf16(float f) { return float_to_bf16(f); }

/* ------------------------------------------------------------ 3D RoPE, tables
 * [comfyui] architecture table: "3D RoPE, sizes [16, 56, 56], theta 256".
 * Reading: the 128 channels of a head are split into consecutive chunks of 16
 * (time), 56 (height), 56 (width).  Inside an axis chunk of width d, channel pair
 * (2i, 2i+1) is rotated by angle pos * theta^(-2i/d), pos the token's coordinate
 * on that axis.  cos/sin are evaluated in double and rounded once to fp32.
 */
void orc_rope_table(double theta, int32_t d_axis, int32_t n_pos, float *cos_out, float *sin_out)
{
    int32_t half = d_axis / 2;
    for (int32_t p = 0; p < n_pos; ++p) {
        for (int32_t i = 0; i < half; ++i) {
            double omega = pow(theta, -2.0 * (double)i / (double)d_axis);
            double ang = (double)p * omega;
            cos_out[(int64_t)p * half + i] = (float)cos(ang);
            sin_out[(int64_t)p * half + i] = (float)sin(ang);
        }
    }
}

/* Token positions of a segment: T*gh*gw video tokens in (t, h, w) row-major order
 * (t from t0), then n_text text tokens, marked with t = -1 (not rotated). */
void orc_positions(int32_t t0, int32_t T, int32_t gh, int32_t gw, int32_t n_text, int32_t *pos)
{
    int64_t k = 0;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < gh; ++h)
            for (int32_t w = 0; w < gw; ++w, ++k) {
                pos[3 * k + 0] = t0 + t;
                pos[3 * k + 1] = h;
                pos[3 * k + 2] = w;
            }
    for (int32_t j = 0; j < n_text; ++j, ++k) {
        pos[3 * k + 0] = -1;
        pos[3 * k + 1] = -1;
        pos[3 * k + 2] = -1;
    }
}

/* Bit-exact path: BF16 in, BF16 out.  Each pair (x0, x1) -> (x0*c - x1*s, x0*s + x1*c)
 * with every product and sum rounded to fp32 (no FMA), then rounded to BF16.
 * x, y: [n_tok][heads][row] with a token stride of row_stride elements; y may be x.
 * pos: [n_tok][3]; t < 0 marks a text token (copied unchanged). */
void orc_rope_bf16(const uint16_t *x, uint16_t *y, int64_t n_tok, int32_t heads, int64_t row_stride,
                   int32_t head_dim, const int32_t *pos, const int32_t split[3], double theta)
{
    int32_t maxp[3] = {1, 1, 1};
    for (int64_t k = 0; k < n_tok; ++k)
        for (int a = 0; a < 3; ++a)
            if (pos[3 * k + a] + 1 > maxp[a]) maxp[a] = pos[3 * k + a] + 1;
    float *cs[3], *sn[3];
    for (int a = 0; a < 3; ++a) {
        cs[a] = (float *)malloc(sizeof(float) * (size_t)maxp[a] * (size_t)(split[a] / 2));
        sn[a] = (float *)malloc(sizeof(float) * (size_t)maxp[a] * (size_t)(split[a] / 2));
        orc_rope_table(theta, split[a], maxp[a], cs[a], sn[a]);
    }
    for (int64_t k = 0; k < n_tok; ++k) {
        for (int32_t h = 0; h < heads; ++h) {
            const uint16_t *xr = x + k * row_stride + (int64_t)h * head_dim;
            uint16_t *yr = y + k * row_stride + (int64_t)h * head_dim;
            if (pos[3 * k] < 0) {
                if (yr != xr) memcpy(yr, xr, sizeof(uint16_t) * (size_t)head_dim);
                continue;
            }
            int32_t base = 0;
            for (int a = 0; a < 3; ++a) {
                int32_t half = split[a] / 2;
                int32_t p = pos[3 * k + a];
                for (int32_t i = 0; i < half; ++i) {
                    float c = cs[a][(int64_t)p * half + i];
                    float s = sn[a][(int64_t)p * half + i];
                    float x0 = bf16_to_float(xr[base + 2 * i]);
                    float x1 = bf16_to_float(xr[base + 2 * i + 1]);
                    float a0 = x0 * c, b0 = x1 * s;
                    float a1 = x0 * s, b1 = x1 * c;
                    float y0 = a0 - b0;
                    float y1 = a1 + b1;
                    yr[base + 2 * i] = float_to_bf16(y0);
                    yr[base + 2 * i + 1] = float_to_bf16(y1);
                }
                base += split[a];
            }
        }
    }
    for (int a = 0; a < 3; ++a) { free(cs[a]); free(sn[a]); }
}

/* Exact-angle float64 path (same rotation, no table rounding): used to pin the
 * geometry (relative-offset invariance, closed-form angles).  x, y: [n_tok][heads][D]. */
void orc_rope_f64(const double *x, double *y, int64_t n_tok, int32_t heads, int32_t head_dim,
                  const int32_t *pos, const int32_t split[3], double theta)
{
    for (int64_t k = 0; k < n_tok; ++k) {
        for (int32_t h = 0; h < heads; ++h) {
            const double *xr = x + (k * heads + h) * head_dim;
            double *yr = y + (k * heads + h) * head_dim;
            if (pos[3 * k] < 0) {
                for (int32_t d = 0; d < head_dim; ++d) yr[d] = xr[d];
                continue;
            }
            int32_t base = 0;
            for (int a = 0; a < 3; ++a) {
                int32_t half = split[a] / 2;
                for (int32_t i = 0; i < half; ++i) {
                    double ang = (double)pos[3 * k + a] * pow(theta, -2.0 * (double)i / (double)split[a]);
                    double c = cos(ang), s = sin(ang);
                    double x0 = xr[base + 2 * i], x1 = xr[base + 2 * i + 1];
                    yr[base + 2 * i] = x0 * c - x1 * s;
                    yr[base + 2 * i + 1] = x0 * s + x1 * c;
                }
                base += split[a];
            }
        }
    }
}

/* ------------------------------------------------------------- INT8 quantise
 * [comfyui] "单张 4090 配置": cached keys and values are stored as INT8.
 * Rule: per token and head, a = max |x| over the 128 channels (x = BF16 value as
 * fp32); scale = fl32(a / 127); a == 0 -> scale 0 and all codes 0; otherwise
 * q = clamp(round_half_even(fl32(x / scale)), -127, 127).
 * rows: [n_rows][d] BF16; codes [n_rows][d]; scales [n_rows]. */
void orc_quantize_rows(const uint16_t *x, int64_t n_rows, int32_t d, int8_t *codes, float *scales)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *xr = x + r * d;
        float a = 0.0f;
        for (int32_t j = 0; j < d; ++j) {
            float v = fabsf(bf16_to_float(xr[j]));
            if (v > a) a = v;
        }
        if (a == 0.0f) {
            scales[r] = 0.0f;
            memset(codes + r * d, 0, (size_t)d);
            continue;
        }
        float scale = a / 127.0f;
        scales[r] = scale;
        for (int32_t j = 0; j < d; ++j) {
            float qf = bf16_to_float(xr[j]) / scale;
            float q = nearbyintf(qf);          /* default rounding mode: to nearest, ties to even */
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            codes[r * d + j] = (int8_t)q;
        }
    }
}

/* ------------------------------------------------------- append to the cache
 * [huawei] 2.1: each segment's K,V are cached and handed to the next segment.
 * For token k of the segment and head h: K row = BF16(RoPE(K)) (video tokens;
 * text tokens unrotated), quantised; V row quantised without rotation.  Rows are
 * written at cache position length + k of the head-major cache [heads][cap][D]. */
void orc_append(const uint16_t *k, const uint16_t *v, int64_t row_stride, int64_t n_tok,
                int32_t heads, int32_t head_dim, const int32_t *pos, const int32_t split[3], double theta,
                int8_t *ck, int8_t *cv, float *cks, float *cvs, int64_t cap, int64_t length)
{
    uint16_t *kr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n_tok > 0 ? n_tok : 1) * (size_t)heads * head_dim);
    /* rotate into a packed [n_tok][heads][D] copy */
    for (int64_t t = 0; t < n_tok; ++t)
        memcpy(kr + t * heads * head_dim, k + t * row_stride, sizeof(uint16_t) * (size_t)heads * head_dim);
    orc_rope_bf16(kr, kr, n_tok, heads, (int64_t)heads * head_dim, head_dim, pos, split, theta);
    uint16_t *row = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)head_dim);
    for (int64_t t = 0; t < n_tok; ++t) {
        for (int32_t h = 0; h < heads; ++h) {
            int64_t dst = (int64_t)h * cap + length + t;
            orc_quantize_rows(kr + (t * heads + h) * head_dim, 1, head_dim, ck + dst * head_dim, cks + dst);
            memcpy(row, v + t * row_stride + (int64_t)h * head_dim, sizeof(uint16_t) * (size_t)head_dim);
            orc_quantize_rows(row, 1, head_dim, cv + dst * head_dim, cvs + dst);
        }
    }
    free(row);
    free(kr);
}

/* --------------------------------------------------- temporal_context gather
 * [comfyui] "单张 4090 配置": the GPU history is limited to 18 temporal_context-
 * sampled latent frames.  Given the sorted selected frames, packed token j comes
 * from archive token frame_token_offset[frames[j / tpf]] + j % tpf; codes and
 * scales of every head are copied; index_map[j] records the archive token. */
void orc_gather(const int8_t *ak, const int8_t *av, const float *aks, const float *avs, int64_t acap,
                int32_t heads, int32_t head_dim, const int32_t *frame_token_offset, int32_t tpf,
                const int32_t *frames, int32_t n_frames,
                int8_t *dk, int8_t *dv, float *dks, float *dvs, int64_t dcap, int32_t *index_map)
{
    int64_t n = (int64_t)n_frames * tpf;
    for (int64_t j = 0; j < n; ++j) {
        int64_t src = (int64_t)frame_token_offset[frames[j / tpf]] + j % tpf;
        index_map[j] = (int32_t)src;
        for (int32_t h = 0; h < heads; ++h) {
            memcpy(dk + ((int64_t)h * dcap + j) * head_dim, ak + ((int64_t)h * acap + src) * head_dim, (size_t)head_dim);
            memcpy(dv + ((int64_t)h * dcap + j) * head_dim, av + ((int64_t)h * acap + src) * head_dim, (size_t)head_dim);
            dks[(int64_t)h * dcap + j] = aks[(int64_t)h * acap + src];
            dvs[(int64_t)h * dcap + j] = avs[(int64_t)h * acap + src];
        }
    }
}

/* -------------------------------------------------- segment-causal attention
 * [comfyui] "一个世界，分段生成": a segment is denoised while attending to the K/V
 * cache of every earlier segment; attention is causal across segments and never
 * needs a future segment.  Reading: query i of current segment s sees every
 * history key (earlier segments, INT8, dequantised k = code * scale exactly in
 * float64) and the current keys of segments 0..s (bidirectional inside s).
 *   O_i = sum_j softmax_j(q_i . k_j * sm_scale) v_j,   LSE_i = log sum_j exp(q_i . k_j * sm_scale)
 * all in float64.  q, kc, vc: BF16 [Lq][heads][D] with token stride row_stride
 * (q and kc already rotated).  History: [heads][h_cap][D] codes, [heads][h_cap] scales.
 * key_parts: bit 0 = use history keys, bit 1 = use current keys.
 * rows: the query rows to evaluate (NULL = all Lq).  out: [n_rows][heads][D]; lse: [n_rows][heads].
 * Returns 0, or -1 on an invalid argument. */
int orc_seg_attn(int32_t heads, int32_t head_dim,
                 const uint16_t *q, const uint16_t *kc, const uint16_t *vc, int64_t row_stride, int64_t lq,
                 const int32_t *seg_off, int32_t n_seg,
                 const int8_t *hk, const int8_t *hv, const float *hks, const float *hvs, int64_t h_cap, int64_t lh,
                 int32_t key_parts, double sm_scale,
                 const int64_t *rows, int64_t n_rows, double *out, double *lse, int32_t n_threads)
{
    if (n_seg < 1 || seg_off[0] != 0 || seg_off[n_seg] != lq) return -1;
    for (int32_t s = 0; s < n_seg; ++s)
        if (seg_off[s + 1] < seg_off[s]) return -1;
    if (rows == NULL) n_rows = lq;
    int64_t n_items = n_rows * heads;
    int use_h = (key_parts & 1) && lh > 0;
    int use_c = (key_parts & 2) != 0;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(lh + lq + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double *acc = (double *)malloc(sizeof(double) * (size_t)head_dim);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t it = 0; it < n_items; ++it) {
            int64_t ri = it / heads;
            int32_t h = (int32_t)(it % heads);
            int64_t i = rows ? rows[ri] : ri;
            if (i < 0 || i >= lq) { bad = 1; continue; }
            /* segment of query i and the end of the current keys it may see */
            int32_t s = 0;
            while (!(seg_off[s] <= i && i < seg_off[s + 1])) ++s;
            int64_t cur_end = seg_off[s + 1];
            for (int32_t d = 0; d < head_dim; ++d)
                qd[d] = (double)bf16_to_float(q[i * row_stride + (int64_t)h * head_dim + d]);
            /* scores over the visible keys: history 0..lh-1, then current 0..cur_end-1 */
            int64_t nk = 0;
            double m = -INFINITY;
            if (use_h) {
                for (int64_t j = 0; j < lh; ++j) {
                    const int8_t *kr = hk + ((int64_t)h * h_cap + j) * head_dim;
                    double ks = (double)hks[(int64_t)h * h_cap + j];
                    double dot = 0.0;
                    for (int32_t d = 0; d < head_dim; ++d) dot += qd[d] * ((double)kr[d] * ks);
                    sc[nk] = dot * sm_scale;
                    if (sc[nk] > m) m = sc[nk];
                    ++nk;
                }
            }
            if (use_c) {
                for (int64_t j = 0; j < cur_end; ++j) {
                    const uint16_t *kr = kc + j * row_stride + (int64_t)h * head_dim;
                    double dot = 0.0;
                    for (int32_t d = 0; d < head_dim; ++d) dot += qd[d] * (double)bf16_to_float(kr[d]);
                    sc[nk] = dot * sm_scale;
                    if (sc[nk] > m) m = sc[nk];
                    ++nk;
                }
            }
            double *o = out + (ri * heads + h) * head_dim;
            if (nk == 0) {
                for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
                if (lse) lse[ri * heads + h] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int64_t j = 0; j < nk; ++j) {
                sc[j] = exp(sc[j] - m);
                l += sc[j];
            }
            for (int32_t d = 0; d < head_dim; ++d) acc[d] = 0.0;
            int64_t j = 0;
            if (use_h) {
                for (int64_t jj = 0; jj < lh; ++jj, ++j) {
                    const int8_t *vr = hv + ((int64_t)h * h_cap + jj) * head_dim;
                    double vs = (double)hvs[(int64_t)h * h_cap + jj];
                    for (int32_t d = 0; d < head_dim; ++d) acc[d] += sc[j] * ((double)vr[d] * vs);
                }
            }
            if (use_c) {
                for (int64_t jj = 0; jj < cur_end; ++jj, ++j) {
                    const uint16_t *vr = vc + jj * row_stride + (int64_t)h * head_dim;
                    for (int32_t d = 0; d < head_dim; ++d) acc[d] += sc[j] * (double)bf16_to_float(vr[d]);
                }
            }
            for (int32_t d = 0; d < head_dim; ++d) o[d] = acc[d] / l;
            if (lse) lse[ri * heads + h] = m + log(l);
        }
        free(sc);
        free(qd);
        free(acc);
    }
    return bad ? -1 : 0;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
