/*
 * gk_oracle.c -- plain, slow, single-threaded reference ("oracle") for one decode
 * step of paged packed-FP8 GQA attention over a whole layer stack.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources it follows (each function names its own):
 *   [GK]  "GPT-OSS-120B giga-kernel decode", sections "Kernel contract",
 *         "KV-cache layout (per-buffer, HMA-preserving)", "DI wiring (NIXL)"
 *         (region list, landing copy, the N - 1 window rule).
 *   [OCP] OCP 8-bit floating point specification, E4M3 format (the "fn" variant:
 *         no infinities, one NaN pattern per sign, largest finite 448).
 *   [SDPA] scaled dot-product attention, softmax(q.k / sqrt(d)) . v, the plain
 *         definition; [RoPE] rotary position embedding in the rotate-half form.
 *
 * Readings taken where the pages are silent:
 *   R1  K packed layout: the trailing [.., block/2, d, 2] view interleaves tokens
 *       2p and 2p+1 of one channel, so K byte (pb, h, t, e) sits at
 *       ((pb*Hkv + h)*(B/2) + t/2)*(2D) + 2e + (t & 1).  V is never packed:
 *       ((pb*Hkv + h)*B + t)*D + e.                          [GK KV-cache layout]
 *       Unpacked K (k_layout = 1) is the tensor the packed view is taken on,
 *       [.., block, d] like V: ((pb*Hkv + h)*B + t)*D + e.  [GK KV-cache layout,
 *       Kernel contract: packed-ness read from the K rank]
 *   R2  RoPE: rotate-half pairs (e, e + D/2) with the per-sequence cos/sin rows
 *       given as inputs [Bt, D/2].                            [GK Kernel contract]
 *   R3  Quantisation: code = E4M3_rne_satfinite(x / scale), one k and one v scale
 *       per layer; dequantisation = decode(code) * scale.  The K path before
 *       encoding is a fixed IEEE fp32 sequence (no fused multiply-add), so the
 *       written bytes are reproducible bit for bit.
 *   R4  Update indices are flat slots pb*B + t of buffer i/2; inactive rows write
 *       nothing.                                               [GK Kernel contract]
 *   R5  Window: the SWA layer attends to the last W positions including the new
 *       one.  Positions are read in the trimmed table's frame: keys
 *       t in [max(0, pos_w - W + 1), pos_w].  Full layers: keys t in [0, pos].
 *   R6  GQA: q head h uses kv head h / (Hq/Hkv).  Softmax scale 1/sqrt(D).
 *       Inactive rows give zero output.  Optional attention sinks (GPT-OSS; not
 *       on the pages): a per-layer, per-head logit sinks[i][h] (natural units)
 *       joins the softmax denominator and carries no value:
 *       out = sum_t e^(s_t) v_t / (sum_t e^(s_t) + e^(sink)).  NULL = none.
 *   R7  Layer i: even -> SWA (table bt_swa, index upd_swa, position pos_w),
 *       odd -> full (bt_full, upd_full, pos); KV buffer j = i / 2.  [GK Kernel contract]
 *
 * Built with -ffp-contract=off so that every fp32 step is a separately rounded
 * IEEE operation; attention arithmetic is in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t num_layers, batch, num_q_heads, num_kv_heads, head_dim;
    int32_t block_size, num_blocks, window, max_blocks_full, max_blocks_swa;
    int32_t k_layout; /* 0: packed K view, 1: unpacked K (laid out like V) */
} ora_shape;

/* ------------------------------------------------------------------------- */
/* E4M3 codec [OCP]                                                           */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code: sign bit, 4-bit exponent field with bias 7, 3-bit
 * mantissa.  Exponent field 0 holds subnormals m * 2^-9; S.1111.111 is NaN;
 * there are no infinities. */
double ora_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, ef = (c >> 3) & 15, m = c & 7;
    double v;
    if (ef == 15 && m == 7)
        return NAN;
    if (ef == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, ef - 7);
    return s ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even mantissa, saturating: |x| > 448
 * gives +-448.  NaN gives 0x7F.  The sign of zero is kept. */
uint8_t ora_e4m3_encode(float xf)
{
    double x = (double)xf, a;
    uint8_t sign;
    int code;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs(x);
    if (a > 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: representable values are n * 2^-9, n = 0..7; n = 8
         * is the smallest normal (code 0x08), so the integer n is the code. */
        code = (int)nearbyint(a * 512.0);
    } else {
        /* a in [2^ex, 2^(ex+1)): spacing 2^(ex-3); n = a / spacing in [8, 16].
         * code = 8*(ex+7) + (n-8); n == 16 carries into the next exponent. */
        int e2;
        double n;
        frexp(a, &e2);
        n = nearbyint(ldexp(a, 3 - (e2 - 1)));
        code = 8 * ((e2 - 1) + 7) + ((int)n - 8);
    }
    if (code > 0x7E)
        code = 0x7E;
    return (uint8_t)(sign | code);
}

void ora_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_e4m3_encode(x[i]);
}

void ora_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------- */
/* bf16 <-> wider types                                                       */
/* ------------------------------------------------------------------------- */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a double to the nearest bf16 value (8 significant bits, ties to even),
 * returned as a double.  Used only to state the tolerance against the bf16
 * output format. */
double ora_round_bf16(double x)
{
    int e;
    double m;
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    m = frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
    if (e < -125) {   /* bf16 subnormal: spacing 2^-133 */
        return ldexp(nearbyint(ldexp(x, 133)), -133);
    }
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

void ora_round_bf16_array(const double *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_round_bf16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Layout: packed K and plain V byte offsets [GK KV-cache layout], reading R1 */
/* ------------------------------------------------------------------------- */

int64_t ora_k_offset(int32_t Hkv, int32_t B, int32_t D, int64_t pb, int32_t h, int32_t t, int32_t e)
{
    int64_t pair_row = (pb * Hkv + h) * (int64_t)(B / 2) + t / 2;
    return pair_row * (2 * (int64_t)D) + 2 * (int64_t)e + (t & 1);
}

int64_t ora_v_offset(int32_t Hkv, int32_t B, int32_t D, int64_t pb, int32_t h, int32_t t, int32_t e)
{
    return ((pb * Hkv + h) * (int64_t)B + t) * (int64_t)D + e;
}

/* Byte of K element (pb, h, t, e) in the shape's K layout. */
static int64_t k_byte(const ora_shape *sh, int64_t pb, int32_t h, int32_t t, int32_t e)
{
    if (sh->k_layout == 0)
        return ora_k_offset(sh->num_kv_heads, sh->block_size, sh->head_dim, pb, h, t, e);
    return ora_v_offset(sh->num_kv_heads, sh->block_size, sh->head_dim, pb, h, t, e);
}

/* Per-layer resources by parity [GK Kernel contract], reading R7. */
static int layer_is_swa(int32_t i) { return (i % 2) == 0; }

/* ------------------------------------------------------------------------- */
/* RoPE [RoPE], reading R2                                                    */
/* ------------------------------------------------------------------------- */

/* The fp32 sequence used for k before quantisation: every product and sum is
 * one IEEE single-precision rounding, no contraction.
 *   x'_e      = (x_e * c_e) - (x_{e+D/2} * s_e)
 *   x'_{e+D/2} = (x_{e+D/2} * c_e) + (x_e * s_e)                              */
void ora_rope_f32(const float *x, const float *cs, const float *sn, int32_t D, float *out)
{
    int32_t half = D / 2;
    for (int32_t e = 0; e < half; ++e) {
        float a = x[e], b = x[e + half];
        float ac = a * cs[e], bs = b * sn[e], bc = b * cs[e], as = a * sn[e];
        out[e] = ac - bs;
        out[e + half] = bc + as;
    }
}

/* Same rotation in double (used for q, whose rotation is not quantised). */
void ora_rope_f64(const double *x, const float *cs, const float *sn, int32_t D, double *out)
{
    int32_t half = D / 2;
    for (int32_t e = 0; e < half; ++e) {
        double a = x[e], b = x[e + half], c = (double)cs[e], s = (double)sn[e];
        out[e] = a * c - b * s;
        out[e + half] = b * c + a * s;
    }
}

/* ------------------------------------------------------------------------- */
/* KV append [GK Kernel contract: two KV-update indices], readings R3, R4, R7 */
/* ------------------------------------------------------------------------- */

/* k_new, v_new: bf16 [NL, Bt, Hkv, D];  cos, sin: fp32 [Bt, D/2];
 * k_scale, v_scale: fp32 [NL];  upd_full, upd_swa: int32 [Bt] flat slots;
 * active: uint8 [Bt];  k_bufs[j], v_bufs[j]: group buffer j's K and V halves.
 * Returns 0, or -1 if a slot lies outside the buffer (nothing is written for it). */
int ora_kv_append(const ora_shape *sh, const uint16_t *k_new, const uint16_t *v_new,
                  const float *cosb, const float *sinb, const float *k_scale, const float *v_scale,
                  const int32_t *upd_full, const int32_t *upd_swa, const uint8_t *active,
                  uint8_t *const *k_bufs, uint8_t *const *v_bufs)
{
    const int32_t NL = sh->num_layers, Bt = sh->batch, Hkv = sh->num_kv_heads, D = sh->head_dim;
    const int32_t B = sh->block_size, half = D / 2;
    int status = 0;
    float *kin = (float *)malloc(sizeof(float) * D), *kr = (float *)malloc(sizeof(float) * D);
    for (int32_t i = 0; i < NL; ++i) {
        int32_t j = i / 2;
        for (int32_t b = 0; b < Bt; ++b) {
            int64_t slot, pb;
            int32_t t;
            if (!active[b])
                continue;
            slot = layer_is_swa(i) ? upd_swa[b] : upd_full[b];
            if (slot < 0 || slot >= (int64_t)sh->num_blocks * B) {
                status = -1;
                continue;
            }
            pb = slot / B;
            t = (int32_t)(slot % B);
            for (int32_t h = 0; h < Hkv; ++h) {
                const uint16_t *kr16 = k_new + (((int64_t)i * Bt + b) * Hkv + h) * D;
                const uint16_t *vr16 = v_new + (((int64_t)i * Bt + b) * Hkv + h) * D;
                for (int32_t e = 0; e < D; ++e)
                    kin[e] = bf16_to_f32(kr16[e]);
                ora_rope_f32(kin, cosb + (int64_t)b * half, sinb + (int64_t)b * half, D, kr);
                for (int32_t e = 0; e < D; ++e) {
                    float kq = kr[e] / k_scale[i];
                    float vq = bf16_to_f32(vr16[e]) / v_scale[i];
                    k_bufs[j][k_byte(sh, pb, h, t, e)] = ora_e4m3_encode(kq);
                    v_bufs[j][ora_v_offset(Hkv, B, D, pb, h, t, e)] = ora_e4m3_encode(vq);
                }
            }
        }
    }
    free(kin);
    free(kr);
    return status;
}

/* ------------------------------------------------------------------------- */
/* Attention for one (layer, sequence, kv head) [SDPA], readings R5, R6, R7   */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q;        /* bf16 [NL, Bt, Hq, D] */
    const uint8_t *kbuf;      /* K half of group buffer i/2 */
    const uint8_t *vbuf;      /* V half of group buffer i/2 */
    const float *k_scale, *v_scale;
    const float *cosb, *sinb; /* [Bt, D/2] */
    const int32_t *bt_full, *bt_swa; /* [Bt, MBF], [Bt, MBS] */
    const int32_t *pos, *pos_w;
    const uint8_t *active;
    const float *sinks;       /* [NL, Hq] or NULL */
} ora_attn_inputs;

/* Key range [lo, hi] (inclusive, in the chosen table's frame) and table row. */
static void key_range(const ora_shape *sh, const ora_attn_inputs *in, int32_t i, int32_t b,
                      int64_t *lo, int64_t *hi, const int32_t **row, int32_t *row_len)
{
    if (layer_is_swa(i)) {
        int64_t pw = in->pos_w[b];
        *lo = pw - sh->window + 1;
        if (*lo < 0)
            *lo = 0;
        *hi = pw;
        *row = in->bt_swa + (int64_t)b * sh->max_blocks_swa;
        *row_len = sh->max_blocks_swa;
    } else {
        *lo = 0;
        *hi = in->pos[b];
        *row = in->bt_full + (int64_t)b * sh->max_blocks_full;
        *row_len = sh->max_blocks_full;
    }
}

/* q' for the G heads of kv head kvh, in double, rotated; [G][D]. */
static void rotated_q(const ora_shape *sh, const ora_attn_inputs *in, int32_t i, int32_t b, int32_t kvh,
                      double *qr)
{
    const int32_t Hq = sh->num_q_heads, D = sh->head_dim, G = Hq / sh->num_kv_heads;
    double *qd = (double *)malloc(sizeof(double) * D);
    for (int32_t g = 0; g < G; ++g) {
        int32_t h = kvh * G + g;
        const uint16_t *qrow = in->q + (((int64_t)i * sh->batch + b) * Hq + h) * D;
        for (int32_t e = 0; e < D; ++e)
            qd[e] = (double)bf16_to_f32(qrow[e]);
        ora_rope_f64(qd, in->cosb + (int64_t)b * (D / 2), in->sinb + (int64_t)b * (D / 2), D, qr + (int64_t)g * D);
    }
    free(qd);
}

/* Dequantised key / value row of token t in the given table frame. */
static int load_kv(const ora_shape *sh, const ora_attn_inputs *in, int32_t i, int32_t kvh,
                   const int32_t *row, int32_t row_len, int64_t t, double *k, double *v)
{
    const int32_t B = sh->block_size, D = sh->head_dim, Hkv = sh->num_kv_heads;
    int64_t blk = t / B;
    int64_t pb;
    int32_t off = (int32_t)(t % B);
    if (blk >= row_len)
        return -1;
    pb = row[blk];
    if (pb < 0 || pb >= sh->num_blocks)
        return -1;
    for (int32_t e = 0; e < D; ++e) {
        k[e] = ora_e4m3_decode(in->kbuf[k_byte(sh, pb, kvh, off, e)]) * (double)in->k_scale[i];
        v[e] = ora_e4m3_decode(in->vbuf[ora_v_offset(Hkv, B, D, pb, kvh, off, e)]) * (double)in->v_scale[i];
    }
    return 0;
}

/* Two-pass softmax attention over keys [lo, hi] split into `nsplit` contiguous
 * chunks.  nsplit == 1 is the plain definition.  For nsplit > 1 each chunk
 * keeps (m_s, l_s, o_s) and the chunks are merged with
 *     M = max m_s,  out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s,
 * the flash-decoding combine; both must agree to rounding.
 * out: [G][D] doubles.  Returns 0 or -1 on an out-of-range table entry. */
int ora_attn_one(const ora_shape *sh, const ora_attn_inputs *in, int32_t i, int32_t b, int32_t kvh,
                 int32_t nsplit, double *out)
{
    const int32_t D = sh->head_dim, G = sh->num_q_heads / sh->num_kv_heads;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    int64_t lo, hi, n, t;
    const int32_t *row;
    int32_t row_len, status = 0;
    double *qr, *kk, *vv, *sc, *ms, *ls, *os;

    memset(out, 0, sizeof(double) * (size_t)G * D);
    if (!in->active[b])
        return 0;
    key_range(sh, in, i, b, &lo, &hi, &row, &row_len);
    n = hi - lo + 1;
    if (n <= 0)
        return 0;
    if (nsplit < 1)
        nsplit = 1;
    if (nsplit > n)
        nsplit = (int32_t)n;

    qr = (double *)malloc(sizeof(double) * G * D);
    kk = (double *)malloc(sizeof(double) * D);
    vv = (double *)malloc(sizeof(double) * D);
    sc = (double *)malloc(sizeof(double) * (size_t)n * G);
    ms = (double *)malloc(sizeof(double) * (size_t)nsplit * G);
    ls = (double *)malloc(sizeof(double) * (size_t)nsplit * G);
    os = (double *)calloc((size_t)nsplit * G * D, sizeof(double));
    rotated_q(sh, in, i, b, kvh, qr);

    /* pass 1: scores */
    for (t = lo; t <= hi; ++t) {
        if (load_kv(sh, in, i, kvh, row, row_len, t, kk, vv) != 0) {
            status = -1;
            for (int32_t g = 0; g < G; ++g)
                sc[(t - lo) * G + g] = -INFINITY;
            continue;
        }
        for (int32_t g = 0; g < G; ++g) {
            double s = 0.0;
            for (int32_t e = 0; e < D; ++e)
                s += qr[(int64_t)g * D + e] * kk[e];
            sc[(t - lo) * G + g] = s * inv_sqrt_d;
        }
    }
    /* per chunk: max, weights, weighted sum of values */
    for (int32_t s = 0; s < nsplit; ++s) {
        int64_t c0 = lo + (n * s) / nsplit, c1 = lo + (n * (s + 1)) / nsplit; /* [c0, c1) */
        for (int32_t g = 0; g < G; ++g) {
            double m = -INFINITY;
            for (t = c0; t < c1; ++t)
                if (sc[(t - lo) * G + g] > m)
                    m = sc[(t - lo) * G + g];
            ms[s * G + g] = m;
            ls[s * G + g] = 0.0;
        }
        for (t = c0; t < c1; ++t) {
            if (load_kv(sh, in, i, kvh, row, row_len, t, kk, vv) != 0)
                continue;
            for (int32_t g = 0; g < G; ++g) {
                double w = exp(sc[(t - lo) * G + g] - ms[s * G + g]);
                ls[s * G + g] += w;
                for (int32_t e = 0; e < D; ++e)
                    os[((int64_t)s * G + g) * D + e] += w * vv[e];
            }
        }
    }
    /* merge (a sink logit joins the denominator with no value) */
    for (int32_t g = 0; g < G; ++g) {
        double M = -INFINITY, L = 0.0, sink = -INFINITY;
        if (in->sinks)
            sink = (double)in->sinks[(int64_t)i * sh->num_q_heads + (int64_t)kvh * G + g];
        for (int32_t s = 0; s < nsplit; ++s)
            if (ms[s * G + g] > M)
                M = ms[s * G + g];
        if (sink > M)
            M = sink;
        for (int32_t s = 0; s < nsplit; ++s)
            L += exp(ms[s * G + g] - M) * ls[s * G + g];
        if (in->sinks)
            L += exp(sink - M);
        for (int32_t e = 0; e < D; ++e) {
            double acc = 0.0;
            for (int32_t s = 0; s < nsplit; ++s)
                acc += exp(ms[s * G + g] - M) * os[((int64_t)s * G + g) * D + e];
            out[(int64_t)g * D + e] = acc / L;
        }
    }
    free(qr);
    free(kk);
    free(vv);
    free(sc);
    free(ms);
    free(ls);
    free(os);
    return status;
}

/* Whole decode-attention step: out [NL, Bt, Hq, D] in double.
 * k_bufs / v_bufs: one pointer per group buffer (NL/2 of them). */
int ora_decode_attn_stack(const ora_shape *sh, const uint16_t *q, const uint8_t *const *k_bufs,
                          const uint8_t *const *v_bufs, const float *k_scale, const float *v_scale,
                          const float *cosb, const float *sinb, const int32_t *bt_full, const int32_t *bt_swa,
                          const int32_t *pos, const int32_t *pos_w, const uint8_t *active,
                          const float *sinks, double *out)
{
    const int32_t NL = sh->num_layers, Bt = sh->batch, Hq = sh->num_q_heads, Hkv = sh->num_kv_heads;
    const int32_t D = sh->head_dim, G = Hq / Hkv;
    int status = 0;
    ora_attn_inputs in;
    in.q = q;
    in.k_scale = k_scale;
    in.v_scale = v_scale;
    in.cosb = cosb;
    in.sinb = sinb;
    in.bt_full = bt_full;
    in.bt_swa = bt_swa;
    in.pos = pos;
    in.pos_w = pos_w;
    in.active = active;
    in.sinks = sinks;
    for (int32_t i = 0; i < NL; ++i) {
        in.kbuf = k_bufs[i / 2];
        in.vbuf = v_bufs[i / 2];
        for (int32_t b = 0; b < Bt; ++b)
            for (int32_t kvh = 0; kvh < Hkv; ++kvh) {
                double *o = out + ((((int64_t)i * Bt + b) * Hq) + (int64_t)kvh * G) * D;
                if (ora_attn_one(sh, &in, i, b, kvh, 1, o) != 0)
                    status = -1;
            }
    }
    return status;
}

/* One (layer, sequence, kv head) with explicit buffers, for sampled checks on
 * large workloads and for the split-invariance check.  out: [G][D]. */
int ora_attn_one_ex(const ora_shape *sh, const uint16_t *q, const uint8_t *kbuf, const uint8_t *vbuf,
                    const float *k_scale, const float *v_scale, const float *cosb, const float *sinb,
                    const int32_t *bt_full, const int32_t *bt_swa, const int32_t *pos, const int32_t *pos_w,
                    const uint8_t *active, const float *sinks, int32_t layer, int32_t b, int32_t kvh,
                    int32_t nsplit, double *out)
{
    ora_attn_inputs in;
    in.q = q;
    in.kbuf = kbuf;
    in.vbuf = vbuf;
    in.k_scale = k_scale;
    in.v_scale = v_scale;
    in.cosb = cosb;
    in.sinb = sinb;
    in.bt_full = bt_full;
    in.bt_swa = bt_swa;
    in.pos = pos;
    in.pos_w = pos_w;
    in.active = active;
    in.sinks = sinks;
    return ora_attn_one(sh, &in, layer, b, kvh, nsplit, out);
}

/* ------------------------------------------------------------------------- */
/* DI landing [GK DI wiring (NIXL)]                                           */
/* ------------------------------------------------------------------------- */

/* Regions of a per-layer binding: layers in order, each contributing its K
 * half and then its V half unless that base address is already a region
 * (paired layers share one group buffer).  bases_k/bases_v: NL addresses as
 * integers.  out: room for 2*NL entries.  Returns the region count. */
int32_t ora_kv_regions(int32_t NL, const uint64_t *bases_k, const uint64_t *bases_v, uint64_t *out)
{
    int32_t n = 0;
    for (int32_t i = 0; i < NL; ++i) {
        uint64_t two[2];
        two[0] = bases_k[i];
        two[1] = bases_v[i];
        for (int h = 0; h < 2; ++h) {
            int seen = 0;
            for (int32_t k = 0; k < n; ++k)
                if (out[k] == two[h])
                    seen = 1;
            if (!seen)
                out[n++] = two[h];
        }
    }
    return n;
}

/* The landing copy: descriptor d moves block_len bytes from src + d*block_len
 * to block dst_block[d] of region dst_region[d], i.e. to
 * region_base + dst_block[d]*block_len.  regions[r] points at region r's
 * bytes (nblocks[r] blocks).  A descriptor out of range is skipped; returns
 * the number skipped. */
int64_t ora_kv_ingest(uint8_t *const *regions, const int64_t *nblocks, int32_t n_regions,
                      int64_t block_len, const int32_t *dst_region, const int32_t *dst_block,
                      int64_t n, const uint8_t *src)
{
    int64_t skipped = 0;
    for (int64_t d = 0; d < n; ++d) {
        int32_t r = dst_region[d], b = dst_block[d];
        if (r < 0 || r >= n_regions || b < 0 || b >= nblocks[r]) {
            ++skipped;
            continue;
        }
        for (int64_t x = 0; x < block_len; ++x)
            regions[r][(int64_t)b * block_len + x] = src[d * block_len + x];
    }
    return skipped;
}

/* Blocks a decode engine needs for a prompt of N tokens when both engines
 * operate at N - 1 (the sliding-window DI truncation fix): the decode step
 * recomputes position N - 1, so keys 0 .. N-2 are transferred.  Full layers
 * hold them in row blocks 0 .. ceil((N-1)/B) - 1; a window layer attends from
 * position N - 1 to keys max(0, N-W) .. N-1, of which N-1 is recomputed, so it
 * needs the blocks of keys max(0, N-W) .. N-2. */
void ora_di_blocks(int64_t N, int32_t B, int32_t W, int64_t *full_count, int64_t *swa_first,
                   int64_t *swa_count)
{
    int64_t first_key = N - W > 0 ? N - W : 0;
    int64_t last_key = N - 2;
    *full_count = (N - 1 + B - 1) / B;
    *swa_first = first_key / B;
    *swa_count = last_key >= first_key ? last_key / B - first_key / B + 1 : 0;
}
