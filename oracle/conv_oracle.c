/*
 * conv_oracle.c -- plain, slow, obviously correct CPU oracle for the forward
 * implicit-GEMM convolution (conv3d over NDHWC activations and KTRSC weights)
 * and for the NCDHW -> NDHWC (+ fp8-e4m3) pack.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Sources followed (pages of the method):
 *  - FlyDSL PR #860 "fp8 conv3d: 8-wave GEMM pipeline + BIG_IN fix", PR summary:
 *    the conv is a GEMM with M = output positions, N = K filters and a
 *    reduction over crs = C*T*R*S; the weight is a plain KTRSC (k, crs) matrix;
 *    the fp8 inputs are E4M3FN; correctness is judged against an fp8-cast
 *    convolution reference, i.e. the convolution of the decoded fp8 values.
 *  - FlyDSL PR #860, commit "temporal fast decode ... verified vs
 *    torch.nn.functional.conv3d": the conv semantics are torch's
 *    (cross-correlation, symmetric zero padding, floor output size).
 *  - FlyDSL PR #860, commit adding the NCDHW->NDHWC fp8 pack kernel: the pack
 *    is a layout transpose plus per-tensor fp8 quantisation.
 *
 * Everything is computed in fp64 from the exact decoded input values and the
 * result is NOT rounded to bf16.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* element decoders (exact)                                            */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; decoding is exact. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3FN (OCP 8-bit float, "FN" = finite + NaN only): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits.  Exponent field 0 encodes subnormals
 * m * 2^-9; the pattern S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Encode a binary32 value to E4M3FN with round-to-nearest, ties to the even
 * code, and saturation to the largest finite magnitude (448 = 0x7E).
 * Written as a nearest-point search over the 127 non-negative finite codes:
 * codes 0x00..0x7E decode to a strictly increasing sequence, so "even code"
 * is "even mantissa" and the search is plain round-to-nearest-even. */
uint8_t oracle_f32_to_e4m3(float v)
{
    double a, lo_v, hi_v, d_lo, d_hi;
    int lo, hi, mid, code;
    uint8_t sign;
    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* largest code with decode(code) <= a */
    lo = 0;
    hi = 0x7E;
    while (lo < hi) {
        mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_to_f64((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    lo_v = oracle_e4m3_to_f64((uint8_t)lo);
    if (lo_v == a)
        return (uint8_t)(sign | lo);
    hi_v = oracle_e4m3_to_f64((uint8_t)(lo + 1));
    d_lo = a - lo_v;
    d_hi = hi_v - a;
    if (d_lo < d_hi)
        code = lo;
    else if (d_hi < d_lo)
        code = lo + 1;
    else
        code = (lo % 2 == 0) ? lo : lo + 1;
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------ */
/* per-tensor fp8 quantisation                                          */
/* ------------------------------------------------------------------ */

/* amax = max |x| over all elements (exact, order free), returned as the
 * binary32 value it is (every bf16 is exactly a binary32). */
float oracle_amax_bf16(const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    int64_t i;
#pragma omp parallel for reduction(max : amax) schedule(static)
    for (i = 0; i < n; ++i) {
        float a = (float)fabs(oracle_bf16_to_f64(x[i]));
        if (a > amax)
            amax = a;
    }
    return amax;
}

/* scale = amax / 448 in binary32 (IEEE division, round to nearest); an
 * all-zero tensor gets scale 1 so that every code is 0.  The scale is a
 * dequantisation multiplier: x ~= decode(q) * scale. */
float oracle_fp8_scale(float amax)
{
    volatile float num = amax, den = 448.0f;
    if (amax == 0.0f)
        return 1.0f;
    return num / den;
}

/* q = E4M3FN_satfinite_rne(binary32(x) / scale), binary32 IEEE division. */
uint8_t oracle_quantize_e4m3(uint16_t xbits, float scale)
{
    uint32_t u = (uint32_t)xbits << 16;
    float f;
    volatile float q;
    memcpy(&f, &u, sizeof f);
    q = f / scale;
    return oracle_f32_to_e4m3(q);
}

/* ------------------------------------------------------------------ */
/* pack: NCDHW -> NDHWC                                                 */
/* ------------------------------------------------------------------ */

/* out[n,d,h,w,c] = in[n,c,d,h,w] (a bit copy). dims = {N, C, D, H, W}. */
void oracle_pack_ncdhw_to_ndhwc_bf16(const uint16_t *in, const int64_t dims[5], uint16_t *out)
{
    int64_t N = dims[0], C = dims[1], S = dims[2] * dims[3] * dims[4];
    int64_t n;
    for (n = 0; n < N; ++n) {
        int64_t s;
#pragma omp parallel for schedule(static)
        for (s = 0; s < S; ++s) {
            int64_t c;
            for (c = 0; c < C; ++c)
                out[(n * S + s) * C + c] = in[(n * C + c) * S + s];
        }
    }
}

/* The fp8 pack: amax over the whole tensor, scale = amax/448, then
 * out[n,d,h,w,c] = q(in[n,c,d,h,w]).  *scale_out receives the scale. */
void oracle_pack_ncdhw_to_ndhwc_fp8(const uint16_t *in, const int64_t dims[5], uint8_t *out,
                                    float *scale_out)
{
    int64_t N = dims[0], C = dims[1], S = dims[2] * dims[3] * dims[4];
    float scale = oracle_fp8_scale(oracle_amax_bf16(in, N * C * S));
    int64_t n;
    for (n = 0; n < N; ++n) {
        int64_t s;
#pragma omp parallel for schedule(static)
        for (s = 0; s < S; ++s) {
            int64_t c;
            for (c = 0; c < C; ++c)
                out[(n * S + s) * C + c] = oracle_quantize_e4m3(in[(n * C + c) * S + s], scale);
        }
    }
    *scale_out = scale;
}

/* ------------------------------------------------------------------ */
/* direct convolution                                                  */
/* ------------------------------------------------------------------ */

enum { ORACLE_ELEM_BF16 = 0, ORACLE_ELEM_E4M3 = 1, ORACLE_ELEM_F64 = 2 };

static double load_elem(const void *base, int64_t i, int elem)
{
    switch (elem) {
    case ORACLE_ELEM_BF16:
        return oracle_bf16_to_f64(((const uint16_t *)base)[i]);
    case ORACLE_ELEM_E4M3:
        return oracle_e4m3_to_f64(((const uint8_t *)base)[i]);
    default:
        return ((const double *)base)[i];
    }
}

/* Output extent of one spatial dimension (floor division, torch semantics). */
int64_t oracle_out_extent(int64_t in, int64_t filt, int stride, int pad, int dil)
{
    int64_t span = in + 2 * (int64_t)pad - (int64_t)dil * (filt - 1) - 1;
    if (span < 0)
        return 0;
    return span / stride + 1;
}

typedef struct {
    int64_t N, D, H, W, C;       /* x extents */
    int64_t xn, xd, xh, xw, xc;  /* x element strides: NDHWC, or NCDHW */
    int64_t K, T, R, S;          /* w: KTRSC (C shared) */
    int64_t Do, Ho, Wo;          /* out: N Do Ho Wo K */
    int sd, sh, sw, pd, ph, pw, dd, dh, dw;
} conv_geom;

static int make_geom(conv_geom *g, const int64_t xd[5], const int64_t wd[5], const int stride[3],
                     const int pad[3], const int dil[3])
{
    g->N = xd[0]; g->D = xd[1]; g->H = xd[2]; g->W = xd[3]; g->C = xd[4];
    g->xc = 1; g->xw = g->C; g->xh = g->W * g->C; g->xd = g->H * g->W * g->C;
    g->xn = g->D * g->H * g->W * g->C;
    g->K = wd[0]; g->T = wd[1]; g->R = wd[2]; g->S = wd[3];
    if (wd[4] != xd[4])
        return -1;
    g->sd = stride[0]; g->sh = stride[1]; g->sw = stride[2];
    g->pd = pad[0]; g->ph = pad[1]; g->pw = pad[2];
    g->dd = dil[0]; g->dh = dil[1]; g->dw = dil[2];
    g->Do = oracle_out_extent(g->D, g->T, g->sd, g->pd, g->dd);
    g->Ho = oracle_out_extent(g->H, g->R, g->sh, g->ph, g->dh);
    g->Wo = oracle_out_extent(g->W, g->S, g->sw, g->pw, g->dw);
    return 0;
}

/* One output element, straight from the definition:
 *   y[n,od,oh,ow,k] = sum_{t,r,s,c} x[n, od*sd-pd+t*dd, oh*sh-ph+r*dh,
 *                                      ow*sw-pw+s*dw, c] * w[k,t,r,s,c]
 * with x = 0 outside the input volume (zero padding, no filter flip). */
static double conv_point(const conv_geom *g, const void *x, const void *w, int elem, int64_t n,
                         int64_t od, int64_t oh, int64_t ow, int64_t k)
{
    double acc = 0.0;
    int64_t t, r, s, c;
    for (t = 0; t < g->T; ++t) {
        int64_t id = od * g->sd - g->pd + t * g->dd;
        if (id < 0 || id >= g->D)
            continue;
        for (r = 0; r < g->R; ++r) {
            int64_t ih = oh * g->sh - g->ph + r * g->dh;
            if (ih < 0 || ih >= g->H)
                continue;
            for (s = 0; s < g->S; ++s) {
                int64_t iw = ow * g->sw - g->pw + s * g->dw;
                int64_t xrow, wrow;
                if (iw < 0 || iw >= g->W)
                    continue;
                xrow = n * g->xn + id * g->xd + ih * g->xh + iw * g->xw;
                wrow = (((k * g->T + t) * g->R + r) * g->S + s) * g->C;
                for (c = 0; c < g->C; ++c)
                    acc += load_elem(x, xrow + c * g->xc, elem) * load_elem(w, wrow + c, elem);
            }
        }
    }
    return acc;
}

/* Full forward convolution.  x NDHWC, w KTRSC, out NDHWC [N,Do,Ho,Wo,K] fp64.
 * The result is scale_x * scale_w * (the exact sum); elem selects how x and w
 * are decoded (bf16 bits, e4m3 bytes or fp64).  Returns 0, or -1 on a shape
 * error. */
int oracle_conv3d_fwd(const void *x, const int64_t xd[5], const void *w, const int64_t wd[5],
                      const int stride[3], const int pad[3], const int dil[3], int elem,
                      double scale_x, double scale_w, double *out)
{
    conv_geom g;
    int64_t rows, m;
    if (make_geom(&g, xd, wd, stride, pad, dil) != 0)
        return -1;
    rows = g.N * g.Do * g.Ho * g.Wo;
#pragma omp parallel for schedule(dynamic, 16)
    for (m = 0; m < rows; ++m) {
        int64_t ow = m % g.Wo, oh = (m / g.Wo) % g.Ho, od = (m / (g.Wo * g.Ho)) % g.Do;
        int64_t n = m / (g.Wo * g.Ho * g.Do), k;
        for (k = 0; k < g.K; ++k)
            out[m * g.K + k] = scale_x * scale_w * conv_point(&g, x, w, elem, n, od, oh, ow, k);
    }
    return 0;
}

/* The same definition evaluated only at the given flat NDHWC output indices. */
static int fwd_points(const conv_geom *gp, const void *x, const void *w, int elem, double scale_x,
                      double scale_w, const int64_t *idx, int64_t n_idx, double *vals);

int oracle_conv3d_fwd_points(const void *x, const int64_t xd[5], const void *w,
                             const int64_t wd[5], const int stride[3], const int pad[3],
                             const int dil[3], int elem, double scale_x, double scale_w,
                             const int64_t *idx, int64_t n_idx, double *vals)
{
    conv_geom g;
    if (make_geom(&g, xd, wd, stride, pad, dil) != 0)
        return -1;
    return fwd_points(&g, x, w, elem, scale_x, scale_w, idx, n_idx, vals);
}

/* The same, with x stored channel-major: x[n,c,d,h,w] at
 * (((n*C + c)*D + d)*H + h)*W + w, xd = {N, C, D, H, W} (torch's own layout);
 * the output indices are still flat NDHWC [N,Do,Ho,Wo,K]. */
int oracle_conv3d_fwd_points_ncdhw(const void *x, const int64_t xd[5], const void *w,
                                   const int64_t wd[5], const int stride[3], const int pad[3],
                                   const int dil[3], int elem, double scale_x, double scale_w,
                                   const int64_t *idx, int64_t n_idx, double *vals)
{
    conv_geom g;
    const int64_t nd[5] = {xd[0], xd[2], xd[3], xd[4], xd[1]};
    if (make_geom(&g, nd, wd, stride, pad, dil) != 0)
        return -1;
    g.xw = 1; g.xh = g.W; g.xd = g.H * g.W; g.xc = g.D * g.H * g.W; g.xn = g.C * g.xc;
    return fwd_points(&g, x, w, elem, scale_x, scale_w, idx, n_idx, vals);
}

static int fwd_points(const conv_geom *gp, const void *x, const void *w, int elem, double scale_x,
                      double scale_w, const int64_t *idx, int64_t n_idx, double *vals)
{
    const conv_geom g = *gp;
    int64_t i, total;
    total = g.N * g.Do * g.Ho * g.Wo * g.K;
    for (i = 0; i < n_idx; ++i)
        if (idx[i] < 0 || idx[i] >= total)
            return -1;
#pragma omp parallel for schedule(dynamic, 64)
    for (i = 0; i < n_idx; ++i) {
        int64_t f = idx[i];
        int64_t k = f % g.K, m = f / g.K;
        int64_t ow = m % g.Wo, oh = (m / g.Wo) % g.Ho, od = (m / (g.Wo * g.Ho)) % g.Do;
        int64_t n = m / (g.Wo * g.Ho * g.Do);
        vals[i] = scale_x * scale_w * conv_point(&g, x, w, elem, n, od, oh, ow, k);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* backward passes (MIOpen PR #10912: backward-data and backward-weights  */
/* of the point-output conv; written here for any geometry)              */
/* ------------------------------------------------------------------ */

/* Backward data: the gradient of sum(out * dy) with respect to x,
 *   dx[n,id,ih,iw,c] = sum over (od,oh,ow,t,r,s,k) with
 *       id = od*sd-pd+t*dd, ih = oh*sh-ph+r*dh, iw = ow*sw-pw+s*dw
 *   of dy[n,od,oh,ow,k] * w[k,t,r,s,c].
 * Computed in the scatter form, straight from that sum: every output element
 * and tap adds its products into the input element it read.  dy is
 * [N,Do,Ho,Wo,K], dx [N,D,H,W,C] fp64 (overwritten).  One thread per batch
 * element n (each writes only its own dx[n]). */
int oracle_conv3d_bwd_data(const void *dy, const int64_t xd[5], const void *w, const int64_t wd[5],
                           const int stride[3], const int pad[3], const int dil[3], int elem,
                           double *dx)
{
    conv_geom g;
    int64_t n;
    if (make_geom(&g, xd, wd, stride, pad, dil) != 0)
        return -1;
    memset(dx, 0, (size_t)(g.N * g.D * g.H * g.W * g.C) * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (n = 0; n < g.N; ++n) {
        int64_t od, oh, ow, k, t, r, s, c;
        for (od = 0; od < g.Do; ++od)
            for (oh = 0; oh < g.Ho; ++oh)
                for (ow = 0; ow < g.Wo; ++ow)
                    for (k = 0; k < g.K; ++k) {
                        double gy = load_elem(dy, (((n * g.Do + od) * g.Ho + oh) * g.Wo + ow) * g.K + k, elem);
                        for (t = 0; t < g.T; ++t) {
                            int64_t id = od * g.sd - g.pd + t * g.dd;
                            if (id < 0 || id >= g.D)
                                continue;
                            for (r = 0; r < g.R; ++r) {
                                int64_t ih = oh * g.sh - g.ph + r * g.dh;
                                if (ih < 0 || ih >= g.H)
                                    continue;
                                for (s = 0; s < g.S; ++s) {
                                    int64_t iw = ow * g.sw - g.pw + s * g.dw;
                                    int64_t xrow, wrow;
                                    if (iw < 0 || iw >= g.W)
                                        continue;
                                    xrow = (((n * g.D + id) * g.H + ih) * g.W + iw) * g.C;
                                    wrow = (((k * g.T + t) * g.R + r) * g.S + s) * g.C;
                                    for (c = 0; c < g.C; ++c)
                                        dx[xrow + c] += gy * load_elem(w, wrow + c, elem);
                                }
                            }
                        }
                    }
    }
    return 0;
}

/* Backward weights: the gradient of sum(out * dy) with respect to w,
 *   dw[k,t,r,s,c] = sum over (n,od,oh,ow) of dy[n,od,oh,ow,k] *
 *                   x[n, od*sd-pd+t*dd, oh*sh-ph+r*dh, ow*sw-pw+s*dw, c]
 * (x = 0 outside the input).  dw is [K,T,R,S,C] fp64 (overwritten).  One
 * thread per filter k. */
int oracle_conv3d_bwd_weight(const void *x, const int64_t xd[5], const void *dy,
                             const int64_t wd[5], const int stride[3], const int pad[3],
                             const int dil[3], int elem, double *dw)
{
    conv_geom g;
    int64_t k;
    if (make_geom(&g, xd, wd, stride, pad, dil) != 0)
        return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (k = 0; k < g.K; ++k) {
        int64_t t, r, s, c, n, od, oh, ow;
        for (t = 0; t < g.T; ++t)
            for (r = 0; r < g.R; ++r)
                for (s = 0; s < g.S; ++s)
                    for (c = 0; c < g.C; ++c) {
                        double acc = 0.0;
                        for (n = 0; n < g.N; ++n)
                            for (od = 0; od < g.Do; ++od) {
                                int64_t id = od * g.sd - g.pd + t * g.dd;
                                if (id < 0 || id >= g.D)
                                    continue;
                                for (oh = 0; oh < g.Ho; ++oh) {
                                    int64_t ih = oh * g.sh - g.ph + r * g.dh;
                                    if (ih < 0 || ih >= g.H)
                                        continue;
                                    for (ow = 0; ow < g.Wo; ++ow) {
                                        int64_t iw = ow * g.sw - g.pw + s * g.dw;
                                        if (iw < 0 || iw >= g.W)
                                            continue;
                                        acc += load_elem(dy, (((n * g.Do + od) * g.Ho + oh) * g.Wo + ow) * g.K + k, elem) *
                                               load_elem(x, (((n * g.D + id) * g.H + ih) * g.W + iw) * g.C + c, elem);
                                    }
                                }
                            }
                        dw[(((k * g.T + t) * g.R + r) * g.S + s) * g.C + c] = acc;
                    }
    }
    return 0;
}

/* Number of threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
