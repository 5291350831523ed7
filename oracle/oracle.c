/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the width-sharded Conv2d with
 * halo exchange, and for the pointwise ops of a ConvNeXt block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library; both sides only draw their inputs from the same seeded generator.
 *
 * Sources (the method is described on two web pages about the same work):
 *   [NV]  NVIDIA technical blog, "Perception model training for autonomous
 *         vehicles with tensor parallelism" (NVIDIA + NIO), Korean mirror:
 *         design section (Shard(3)/Replicate placements, the sharding rules of
 *         aten.convolution and aten.convolution_backward, _Partial gradients),
 *         Figure 1 (halo exchange and crop, forward) and Figure 2 (backward).
 *   [KW]  kwkr.cn news/18980, Chinese write-up of the same method: section 2.1
 *         (Shard(3) of (7,3,512,2048) over 4 devices), section 2.2 (halo
 *         exchange / concat / crop, and the zero-pad plus exchange of the
 *         backward pass, _Partial weight gradients reduced across devices),
 *         section 3.2 (the _conv_forward override: exchange, local conv, crop).
 *
 * Convolution conventions (the standard cross-correlation that the pages'
 * aten.convolution computes): NCHW tensors, weight [C_out][C_in/groups][kh][kw],
 * zero padding `padding` on every side, the same stride in H and W, output
 * size (in + 2*padding - k) / stride + 1.
 *
 * Every sum is accumulated in double from the fp32 inputs (fp32 x fp32 products
 * are exact in double) and returned in double.
 *
 * Readings taken where the pages are silent or garbled:
 *   - Halo widths: left = padding, right = the columns the last owned output
 *     of a shard still reads past the shard (k - padding - stride for the
 *     configurations used here).  [NV] only gives the 5x5 / pad 2 / stride 1
 *     example (2 columns from each neighbour).
 *   - Local conv of [KW] 3.2: the printed call passes padding 0 and then crops
 *     `padding` columns on each side, which would drop valid columns.  Read as:
 *     local conv with `padding` in both H and W on the extended tile, then a
 *     crop of padding/stride output columns on the left, keeping the shard's
 *     owned columns (for padding 0 there is neither halo nor crop).  This needs
 *     stride | padding, which holds for every configuration used here.
 *   - Backward ([KW] 2.2, [NV] Figure 2): the shard's grad_output is zero-padded
 *     back to the local conv's output width, the local grad_input is computed
 *     on the extended tile, and the halo columns of that grad_input are sent
 *     back to (accumulated into) the neighbouring shards.  The local
 *     grad_weight / grad_bias are the per-shard _Partial values; their sum over
 *     shards is the full gradient ([NV] design section).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int N, C_in, H, W, C_out, kh, kw, stride, padding, groups, num_shards;
    int num_shards_h; /* row shards (Shard(2)); 0 or 1: none */
} or_desc;

/* Per-shard extent: input columns [in_begin, in_end), halo widths, and the
 * owned output columns [out_begin, out_end). */
typedef struct {
    int in_begin, in_end, halo_left, halo_right, out_begin, out_end;
} or_extent;

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Output size of a convolution along one dimension. */
int or_out_size(int in, int k, int s, int p) {
    if (s <= 0 || k <= 0 || p < 0) return -1;
    int span = in + 2 * p - k;
    if (span < 0) return 0;
    return span / s + 1;
}

static int desc_ok(const or_desc* d) {
    if (d->N < 0 || d->C_in <= 0 || d->H <= 0 || d->W <= 0 || d->C_out <= 0) return 0;
    if (d->kh <= 0 || d->kw <= 0 || d->stride <= 0 || d->padding < 0 || d->groups <= 0) return 0;
    if (d->C_in % d->groups || d->C_out % d->groups) return 0;
    return 1;
}

#define X4(t, C, H, W, n, c, h, w) (t)[(((int64_t)(n) * (C) + (c)) * (H) + (h)) * (int64_t)(W) + (w)]
#define W4(t, Cg, kh, kw, co, ci, u, v) (t)[(((int64_t)(co) * (Cg) + (ci)) * (kh) + (u)) * (kw) + (v)]

/* ---------------------------------------------------------------------------
 * Unsharded convolution: the plain definition.
 * ------------------------------------------------------------------------- */

/* y[n,co,i,j] = b[co] + sum_{ci',u,v} w[co,ci',u,v] * x[n, g*Cg+ci', i*s-p+u, j*s-p+v]
 * with x = 0 outside [0,H) x [0,W).  b may be NULL.  y is [N][C_out][Hout][Wout]. */
int or_conv2d_fwd(const or_desc* d, const float* x, const float* w, const float* b, double* y) {
    if (!desc_ok(d)) return 1;
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int s = d->stride, p = d->padding;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < d->N; n++)
        for (int co = 0; co < d->C_out; co++) {
            const int g = co / Cgo;
            for (int i = 0; i < Ho; i++)
                for (int j = 0; j < Wo; j++) {
                    double acc = b ? (double)b[co] : 0.0;
                    for (int cl = 0; cl < Cgi; cl++) {
                        const int ci = g * Cgi + cl;
                        for (int u = 0; u < d->kh; u++) {
                            const int h = i * s - p + u;
                            if (h < 0 || h >= d->H) continue;
                            for (int v = 0; v < d->kw; v++) {
                                const int c = j * s - p + v;
                                if (c < 0 || c >= d->W) continue;
                                acc += (double)W4(w, Cgi, d->kh, d->kw, co, cl, u, v) *
                                       (double)X4(x, d->C_in, d->H, d->W, n, ci, h, c);
                            }
                        }
                    }
                    X4(y, d->C_out, Ho, Wo, n, co, i, j) = acc;
                }
        }
    return 0;
}

/* grad_input: the transpose of the forward loop.  Every product term
 * w[co,ci',u,v] * x[n,ci,h,c] of the forward sum contributes
 * w[co,ci',u,v] * gy[n,co,i,j] to gx[n,ci,h,c].  gx is [N][C_in][H][W]. */
int or_conv2d_bwd_input(const or_desc* d, const float* w, const float* gy, double* gx) {
    if (!desc_ok(d)) return 1;
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int s = d->stride, p = d->padding;
    memset(gx, 0, sizeof(double) * (size_t)d->N * d->C_in * d->H * d->W);
    /* (n, group) pairs own disjoint slices of gx. */
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < d->N; n++)
        for (int g = 0; g < d->groups; g++)
            for (int co = g * Cgo; co < (g + 1) * Cgo; co++)
                for (int i = 0; i < Ho; i++)
                    for (int j = 0; j < Wo; j++) {
                        const double gv = (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j);
                        for (int cl = 0; cl < Cgi; cl++) {
                            const int ci = g * Cgi + cl;
                            for (int u = 0; u < d->kh; u++) {
                                const int h = i * s - p + u;
                                if (h < 0 || h >= d->H) continue;
                                for (int v = 0; v < d->kw; v++) {
                                    const int c = j * s - p + v;
                                    if (c < 0 || c >= d->W) continue;
                                    X4(gx, d->C_in, d->H, d->W, n, ci, h, c) +=
                                        (double)W4(w, Cgi, d->kh, d->kw, co, cl, u, v) * gv;
                                }
                            }
                        }
                    }
    return 0;
}

/* grad_weight: gw[co,ci',u,v] = sum_{n,i,j} gy[n,co,i,j] * x[n,ci,i*s-p+u,j*s-p+v]. */
int or_conv2d_bwd_weight(const or_desc* d, const float* x, const float* gy, double* gw) {
    if (!desc_ok(d)) return 1;
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int s = d->stride, p = d->padding;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int co = 0; co < d->C_out; co++)
        for (int cl = 0; cl < Cgi; cl++) {
            const int ci = (co / Cgo) * Cgi + cl;
            for (int u = 0; u < d->kh; u++)
                for (int v = 0; v < d->kw; v++) {
                    double acc = 0.0;
                    for (int n = 0; n < d->N; n++)
                        for (int i = 0; i < Ho; i++) {
                            const int h = i * s - p + u;
                            if (h < 0 || h >= d->H) continue;
                            for (int j = 0; j < Wo; j++) {
                                const int c = j * s - p + v;
                                if (c < 0 || c >= d->W) continue;
                                acc += (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j) *
                                       (double)X4(x, d->C_in, d->H, d->W, n, ci, h, c);
                            }
                        }
                    W4(gw, Cgi, d->kh, d->kw, co, cl, u, v) = acc;
                }
        }
    return 0;
}

/* grad_bias: gb[co] = sum_{n,i,j} gy[n,co,i,j]. */
int or_conv2d_bwd_bias(const or_desc* d, const float* gy, double* gb) {
    if (!desc_ok(d)) return 1;
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    for (int co = 0; co < d->C_out; co++) {
        double acc = 0.0;
        for (int n = 0; n < d->N; n++)
            for (int i = 0; i < Ho; i++)
                for (int j = 0; j < Wo; j++) acc += (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j);
        gb[co] = acc;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Single-element evaluators (same definitions, one output at a time), used to
 * check sampled outputs of full-size runs.
 * ------------------------------------------------------------------------- */

double or_conv2d_fwd_at(const or_desc* d, const float* x, const float* w, const float* b,
                        int n, int co, int i, int j) {
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int g = co / Cgo, s = d->stride, p = d->padding;
    double acc = b ? (double)b[co] : 0.0;
    for (int cl = 0; cl < Cgi; cl++)
        for (int u = 0; u < d->kh; u++) {
            const int h = i * s - p + u;
            if (h < 0 || h >= d->H) continue;
            for (int v = 0; v < d->kw; v++) {
                const int c = j * s - p + v;
                if (c < 0 || c >= d->W) continue;
                acc += (double)W4(w, Cgi, d->kh, d->kw, co, cl, u, v) *
                       (double)X4(x, d->C_in, d->H, d->W, n, g * Cgi + cl, h, c);
            }
        }
    return acc;
}

/* gx at one input position, written as a gather: the outputs (i, j) whose
 * window covers (h, c) at tap (u, v) satisfy i*s = h + p - u, j*s = c + p - v. */
double or_conv2d_gx_at(const or_desc* d, const float* w, const float* gy, int n, int ci, int h, int c) {
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int g = ci / Cgi, cl = ci % Cgi, s = d->stride, p = d->padding;
    double acc = 0.0;
    for (int co = g * Cgo; co < (g + 1) * Cgo; co++)
        for (int u = 0; u < d->kh; u++) {
            const int ti = h + p - u;
            if (ti < 0 || ti % s) continue;
            const int i = ti / s;
            if (i >= Ho) continue;
            for (int v = 0; v < d->kw; v++) {
                const int tj = c + p - v;
                if (tj < 0 || tj % s) continue;
                const int j = tj / s;
                if (j >= Wo) continue;
                acc += (double)W4(w, Cgi, d->kh, d->kw, co, cl, u, v) *
                       (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j);
            }
        }
    return acc;
}

/* gw[co,ci',u,v] restricted to output columns [j_begin, j_end): with a
 * shard's owned columns this is that shard's _Partial value. */
double or_conv2d_gw_at(const or_desc* d, const float* x, const float* gy, int co, int cl, int u, int v,
                       int j_begin, int j_end, int i_begin, int i_end) {
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    const int Cgi = d->C_in / d->groups, Cgo = d->C_out / d->groups;
    const int ci = (co / Cgo) * Cgi + cl, s = d->stride, p = d->padding;
    double acc = 0.0;
    for (int n = 0; n < d->N; n++)
        for (int i = i_begin; i < i_end && i < Ho; i++) {
            const int h = i * s - p + u;
            if (h < 0 || h >= d->H) continue;
            for (int j = j_begin; j < j_end && j < Wo; j++) {
                const int c = j * s - p + v;
                if (c < 0 || c >= d->W) continue;
                acc += (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j) *
                       (double)X4(x, d->C_in, d->H, d->W, n, ci, h, c);
            }
        }
    return acc;
}

double or_conv2d_gb_at(const or_desc* d, const float* gy, int co, int j_begin, int j_end) {
    const int Ho = or_out_size(d->H, d->kh, d->stride, d->padding);
    const int Wo = or_out_size(d->W, d->kw, d->stride, d->padding);
    double acc = 0.0;
    for (int n = 0; n < d->N; n++)
        for (int i = 0; i < Ho; i++)
            for (int j = j_begin; j < j_end && j < Wo; j++) acc += (double)X4(gy, d->C_out, Ho, Wo, n, co, i, j);
    return acc;
}

/* ---------------------------------------------------------------------------
 * The sharded method, step by step ([NV] design section, Figures 1-2;
 * [KW] 2.1, 2.2, 3.2).
 * ------------------------------------------------------------------------- */

/* Shard(3) plan: W split into num_shards equal column blocks ([NV] design
 * section; [KW] 2.1).  Shard r owns input columns [r*Wl, (r+1)*Wl) and output
 * columns [r*Wl/s, (r+1)*Wl/s) (the last shard also takes any output columns
 * past W/s).  Halo widths: the columns outside its block that its owned
 * outputs read.  Returns 0, or 2 when the layout is not supported (W not
 * divisible by the shard count, Wl not divisible by the stride, stride not
 * dividing the padding, or a halo wider than a neighbouring shard). */
static int plan_1d(int in, int k, int s, int p, int S, int out, or_extent* ext) {
    if (in % S) return 2;
    const int L = in / S;
    if (L % s || p % s) return 2;
    for (int r = 0; r < S; r++) {
        or_extent e;
        e.in_begin = r * L;
        e.in_end = (r + 1) * L;
        e.out_begin = r * L / s;
        e.out_end = (r == S - 1) ? out : (r + 1) * L / s;
        if (e.out_end > out) e.out_end = out;
        if (e.out_begin > e.out_end) e.out_begin = e.out_end;
        e.halo_left = 0;
        e.halo_right = 0;
        if (e.out_end > e.out_begin) {
            const int first = e.out_begin * s - p;                /* first index read */
            const int last = (e.out_end - 1) * s - p + k - 1;     /* last index read  */
            e.halo_left = first < e.in_begin ? e.in_begin - first : 0;
            e.halo_right = last >= e.in_end ? last - e.in_end + 1 : 0;
        }
        if (e.halo_left > L || e.halo_right > L) return 2;
        ext[r] = e;
    }
    return 0;
}

static int shards_h(const or_desc* d) { return d->num_shards_h > 1 ? d->num_shards_h : 1; }

int or_shard_plan(const or_desc* d, or_extent* ext, int* Ho_out, int* Wo_out) {
    if (!desc_ok(d) || d->num_shards <= 0) return 1;
    const int s = d->stride, p = d->padding;
    const int Ho = or_out_size(d->H, d->kh, s, p), Wo = or_out_size(d->W, d->kw, s, p);
    if (Ho <= 0 || Wo <= 0) return 1;
    const int rc = plan_1d(d->W, d->kw, s, p, d->num_shards, Wo, ext);
    if (rc) return rc;
    if (Ho_out) *Ho_out = Ho;
    if (Wo_out) *Wo_out = Wo;
    return 0;
}

/* Row shards (the pages' Shard(2) variant: [KW] 5.2 switches the sharded
 * dimension to the height at very high resolution): the same rule as the
 * column plan, applied to H with the kernel height.  With num_shards_h <= 1
 * there are no row neighbours: one extent covers every row with no halo rows
 * (the local conv's padding supplies the image edges) and no row crop. */
int or_shard_plan_h(const or_desc* d, or_extent* ext) {
    if (!desc_ok(d)) return 1;
    const int s = d->stride, p = d->padding;
    const int Ho = or_out_size(d->H, d->kh, s, p);
    if (Ho <= 0) return 1;
    if (shards_h(d) == 1) {
        or_extent e = {0, d->H, 0, 0, 0, Ho};
        ext[0] = e;
        return 0;
    }
    return plan_1d(d->H, d->kh, s, p, shards_h(d), Ho, ext);
}

/* Halo exchange + concat for shard q = a * S + b of the row x column shard
 * grid ([KW] 2.2 steps 1-2, applied to rows and columns): the extended tile
 * [N][C][top + Hl + bottom][left + Wl + right] holds the shard's block and the
 * halo rows and columns around it read from the neighbouring shards; positions
 * outside the image are zero. */
int or_halo_extend(const or_desc* d, int q, const float* x, float* x_ext) {
    or_extent ew[1024], eh[1024];
    if (d->num_shards > 1024 || shards_h(d) > 1024) return 1;
    int rc = or_shard_plan(d, ew, NULL, NULL);
    if (!rc) rc = or_shard_plan_h(d, eh);
    if (rc) return rc;
    const or_extent e = ew[q % d->num_shards], f = eh[q / d->num_shards];
    const int We = e.halo_left + (e.in_end - e.in_begin) + e.halo_right;
    const int He = f.halo_left + (f.in_end - f.in_begin) + f.halo_right;
    for (int n = 0; n < d->N; n++)
        for (int c = 0; c < d->C_in; c++)
            for (int r = 0; r < He; r++)
                for (int t = 0; t < We; t++) {
                    const int row = f.in_begin - f.halo_left + r, col = e.in_begin - e.halo_left + t;
                    X4(x_ext, d->C_in, He, We, n, c, r, t) =
                        (row >= 0 && row < d->H && col >= 0 && col < d->W) ? X4(x, d->C_in, d->H, d->W, n, c, row, col)
                                                                           : 0.0f;
                }
    return 0;
}

/* Forward, shard by shard over the row x column grid: exchange + concat, local
 * conv with padding in both H and W on the extended tile, crop to the owned
 * output rows and columns. */
int or_sharded_fwd(const or_desc* d, const float* x, const float* w, const float* b, double* y) {
    or_extent ew[1024], eh[1024];
    int Ho, Wo;
    if (d->num_shards > 1024 || shards_h(d) > 1024) return 1;
    int rc = or_shard_plan(d, ew, &Ho, &Wo);
    if (!rc) rc = or_shard_plan_h(d, eh);
    if (rc) return rc;
    const int s = d->stride, p = d->padding, S = d->num_shards;
    for (int q = 0; q < shards_h(d) * S; q++) {
        const or_extent e = ew[q % S], f = eh[q / S];
        if (e.out_end <= e.out_begin || f.out_end <= f.out_begin) continue;
        const int We = e.halo_left + (e.in_end - e.in_begin) + e.halo_right;
        const int He = f.halo_left + (f.in_end - f.in_begin) + f.halo_right;
        float* xe = (float*)malloc(sizeof(float) * (size_t)d->N * d->C_in * He * We);
        or_halo_extend(d, q, x, xe);
        or_desc ld = *d;
        ld.W = We;
        ld.H = He;
        const int Wloc = or_out_size(We, d->kw, s, p), Hloc = or_out_size(He, d->kh, s, p);
        double* yl = (double*)malloc(sizeof(double) * (size_t)d->N * d->C_out * Hloc * Wloc);
        or_conv2d_fwd(&ld, xe, w, b, yl);
        /* Crop: owned output column out_begin + t reads extended-tile columns
         * from (out_begin*s - p) - (in_begin - halo_left) on; with padding p
         * applied to the tile that is local output column t + crop (rows alike). */
        const int crop = ((e.out_begin * s - p) - (e.in_begin - e.halo_left) + p) / s;
        const int crop_h = ((f.out_begin * s - p) - (f.in_begin - f.halo_left) + p) / s;
        for (int n = 0; n < d->N; n++)
            for (int co = 0; co < d->C_out; co++)
                for (int i = 0; i < f.out_end - f.out_begin; i++)
                    for (int t = 0; t < e.out_end - e.out_begin; t++)
                        X4(y, d->C_out, Ho, Wo, n, co, f.out_begin + i, e.out_begin + t) =
                            X4(yl, d->C_out, Hloc, Wloc, n, co, i + crop_h, t + crop);
        free(yl);
        free(xe);
    }
    return 0;
}

/* Backward, shard by shard over the row x column grid: zero-pad the shard's
 * grad_output to the local conv's output size (undoing the crop), local
 * grad_input / grad_weight / grad_bias on the extended tile, then send the halo
 * rows and columns of the local grad_input back to the shards that own them
 * (accumulate into gx).  gw_part is [Sh*S][C_out][C_in/groups][kh][kw] and
 * gb_part is [Sh*S][C_out], shard q = a * S + b; either may be NULL.  gx (NULL
 * allowed) is [N][C_in][H][W]. */
int or_sharded_bwd(const or_desc* d, const float* x, const float* w, const float* gy,
                   double* gx, double* gw_part, double* gb_part) {
    or_extent ew[1024], eh[1024];
    int Ho, Wo;
    if (d->num_shards > 1024 || shards_h(d) > 1024) return 1;
    int rc = or_shard_plan(d, ew, &Ho, &Wo);
    if (!rc) rc = or_shard_plan_h(d, eh);
    if (rc) return rc;
    const int s = d->stride, p = d->padding, S = d->num_shards;
    const size_t wsz = (size_t)d->C_out * (d->C_in / d->groups) * d->kh * d->kw;
    if (gx) memset(gx, 0, sizeof(double) * (size_t)d->N * d->C_in * d->H * d->W);
    for (int q = 0; q < shards_h(d) * S; q++) {
        const or_extent e = ew[q % S], f = eh[q / S];
        if (e.out_end <= e.out_begin || f.out_end <= f.out_begin) {
            if (gw_part) memset(gw_part + q * wsz, 0, sizeof(double) * wsz);
            if (gb_part) memset(gb_part + (size_t)q * d->C_out, 0, sizeof(double) * d->C_out);
            continue;
        }
        const int We = e.halo_left + (e.in_end - e.in_begin) + e.halo_right;
        const int He = f.halo_left + (f.in_end - f.in_begin) + f.halo_right;
        float* xe = (float*)malloc(sizeof(float) * (size_t)d->N * d->C_in * He * We);
        or_halo_extend(d, q, x, xe);
        or_desc ld = *d;
        ld.W = We;
        ld.H = He;
        const int Wloc = or_out_size(We, d->kw, s, p), Hloc = or_out_size(He, d->kh, s, p);
        const int crop = ((e.out_begin * s - p) - (e.in_begin - e.halo_left) + p) / s;
        const int crop_h = ((f.out_begin * s - p) - (f.in_begin - f.halo_left) + p) / s;
        float* gyl = (float*)calloc((size_t)d->N * d->C_out * Hloc * Wloc, sizeof(float));
        for (int n = 0; n < d->N; n++)
            for (int co = 0; co < d->C_out; co++)
                for (int i = 0; i < f.out_end - f.out_begin; i++)
                    for (int t = 0; t < e.out_end - e.out_begin; t++)
                        X4(gyl, d->C_out, Hloc, Wloc, n, co, i + crop_h, t + crop) =
                            X4(gy, d->C_out, Ho, Wo, n, co, f.out_begin + i, e.out_begin + t);
        if (gx) {
            double* gxe = (double*)malloc(sizeof(double) * (size_t)d->N * d->C_in * He * We);
            or_conv2d_bwd_input(&ld, w, gyl, gxe);
            for (int n = 0; n < d->N; n++)
                for (int c = 0; c < d->C_in; c++)
                    for (int r = 0; r < He; r++)
                        for (int t = 0; t < We; t++) {
                            const int row = f.in_begin - f.halo_left + r, col = e.in_begin - e.halo_left + t;
                            if (row >= 0 && row < d->H && col >= 0 && col < d->W)
                                X4(gx, d->C_in, d->H, d->W, n, c, row, col) += X4(gxe, d->C_in, He, We, n, c, r, t);
                        }
            free(gxe);
        }
        if (gw_part) or_conv2d_bwd_weight(&ld, xe, gyl, gw_part + q * wsz);
        if (gb_part) or_conv2d_bwd_bias(&ld, gyl, gb_part + (size_t)q * d->C_out);
        free(gyl);
        free(xe);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Pointwise ops of a ConvNeXt block (channels-first, shard-local: no halo).
 * Tensors are [N][C][HW]; all in double.
 * ------------------------------------------------------------------------- */

/* LayerNorm over C at every (n, position): mean, biased variance,
 * y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c].
 * mean / rstd ([N][HW]) may be NULL. */
void or_layernorm_c_fwd(int N, int C, int64_t HW, const double* x, const double* gamma, const double* beta,
                        double eps, double* y, double* mean, double* rstd) {
#pragma omp parallel for collapse(2)
    for (int n = 0; n < N; n++)
        for (int64_t q = 0; q < HW; q++) {
            double mu = 0.0, var = 0.0;
            for (int c = 0; c < C; c++) mu += x[((int64_t)n * C + c) * HW + q];
            mu /= C;
            for (int c = 0; c < C; c++) {
                const double t = x[((int64_t)n * C + c) * HW + q] - mu;
                var += t * t;
            }
            var /= C;
            const double rs = 1.0 / sqrt(var + eps);
            for (int c = 0; c < C; c++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                y[o] = (x[o] - mu) * rs * gamma[c] + beta[c];
            }
            if (mean) mean[(int64_t)n * HW + q] = mu;
            if (rstd) rstd[(int64_t)n * HW + q] = rs;
        }
}

/* LayerNorm backward.  With xhat = (x - mean) * rstd and g = gy * gamma:
 * gx = rstd * (g - mean_c(g) - xhat * mean_c(g * xhat)),
 * ggamma[c] = sum gy * xhat, gbeta[c] = sum gy (sums over n and positions). */
void or_layernorm_c_bwd(int N, int C, int64_t HW, const double* x, const double* gamma, const double* gy,
                        double eps, double* gx, double* ggamma, double* gbeta) {
    for (int c = 0; c < C; c++) {
        ggamma[c] = 0.0;
        gbeta[c] = 0.0;
    }
    for (int n = 0; n < N; n++)
        for (int64_t q = 0; q < HW; q++) {
            double mu = 0.0, var = 0.0;
            for (int c = 0; c < C; c++) mu += x[((int64_t)n * C + c) * HW + q];
            mu /= C;
            for (int c = 0; c < C; c++) {
                const double t = x[((int64_t)n * C + c) * HW + q] - mu;
                var += t * t;
            }
            var /= C;
            const double rs = 1.0 / sqrt(var + eps);
            double mg = 0.0, mgx = 0.0;
            for (int c = 0; c < C; c++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                const double xh = (x[o] - mu) * rs;
                const double g = gy[o] * gamma[c];
                mg += g;
                mgx += g * xh;
                ggamma[c] += gy[o] * xh;
                gbeta[c] += gy[o];
            }
            mg /= C;
            mgx /= C;
            for (int c = 0; c < C; c++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                const double xh = (x[o] - mu) * rs;
                gx[o] = rs * (gy[o] * gamma[c] - mg - xh * mgx);
            }
        }
}

/* GELU, exact form: x * Phi(x), Phi(x) = (1 + erf(x / sqrt 2)) / 2. */
void or_gelu_fwd(int64_t n, const double* x, double* y) {
    for (int64_t i = 0; i < n; i++) y[i] = x[i] * 0.5 * (1.0 + erf(x[i] / sqrt(2.0)));
}

/* d/dx GELU = Phi(x) + x * phi(x), phi(x) = exp(-x^2 / 2) / sqrt(2 pi). */
void or_gelu_bwd(int64_t n, const double* x, const double* gy, double* gx) {
    const double inv_sqrt_2pi = 1.0 / sqrt(2.0 * M_PI);
    for (int64_t i = 0; i < n; i++) {
        const double Phi = 0.5 * (1.0 + erf(x[i] / sqrt(2.0)));
        const double phi = exp(-0.5 * x[i] * x[i]) * inv_sqrt_2pi;
        gx[i] = gy[i] * (Phi + x[i] * phi);
    }
}

/* Layer scale and residual: out = res + gamma[c] * branch. */
void or_layerscale_residual_fwd(int N, int C, int64_t HW, const double* res, const double* branch,
                                const double* gamma, double* out) {
    for (int n = 0; n < N; n++)
        for (int c = 0; c < C; c++)
            for (int64_t q = 0; q < HW; q++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                out[o] = res[o] + gamma[c] * branch[o];
            }
}

/* Backward: gres = gy, gbranch = gamma[c] * gy, ggamma[c] = sum branch * gy. */
void or_layerscale_residual_bwd(int N, int C, int64_t HW, const double* branch, const double* gamma,
                                const double* gy, double* gres, double* gbranch, double* ggamma) {
    for (int c = 0; c < C; c++) ggamma[c] = 0.0;
    for (int n = 0; n < N; n++)
        for (int c = 0; c < C; c++)
            for (int64_t q = 0; q < HW; q++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                if (gres) gres[o] = gy[o];
                gbranch[o] = gamma[c] * gy[o];
                ggamma[c] += branch[o] * gy[o];
            }
}

/* DropPath (stochastic depth) with a shard-consistent draw.  [NV] design
 * section: ConvNeXt-XL's DropPath draws a per-sample Bernoulli (aten.bernoulli)
 * that every device must reproduce; [KW] section 3.1 (a distributed DropPath
 * layer keeps the RNG consistent) and section 6.1 (every DropPath layer on every
 * device uses the same seed).
 * Reading: sample n keeps its residual branch with probability 1 - p, a kept
 * branch is scaled by 1 / (1 - p) (stochastic-depth scaling), and the draw for
 * sample n is output number offset + n of a SplitMix64 generator seeded with
 * `seed`: it depends on (seed, offset, n) only, so any device holding sample n
 * draws the same value.  Keep iff the top 24 bits u of that output satisfy
 * u >= floor(p * 2^24) (an integer decision, the same on every side).
 * SplitMix64: G. L. Steele, D. Lea, C. H. Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014, with the finaliser of S. Vigna's
 * public-domain splitmix64.c: output i of the generator seeded with s mixes
 * s + (i + 1) * 0x9E3779B97F4A7C15. */
uint64_t or_splitmix64(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

int or_drop_path_mask(int N, float p, uint64_t seed, uint64_t offset, float* mask) {
    if (N < 0 || !(p >= 0.0f) || !(p < 1.0f)) return 1;
    const uint32_t t = (uint32_t)floor((double)p * 16777216.0);
    const float scale = 1.0f / (1.0f - p);
    for (int n = 0; n < N; n++) {
        const uint32_t u = (uint32_t)(or_splitmix64(seed, offset + (uint64_t)n) >> 40);
        mask[n] = u >= t ? scale : 0.0f;
    }
    return 0;
}

/* Layer scale, DropPath and residual: out = res + mask[n] * gamma[c] * branch. */
void or_layerscale_droppath_fwd(int N, int C, int64_t HW, const double* res, const double* branch,
                                const double* gamma, const double* mask, double* out) {
    for (int n = 0; n < N; n++)
        for (int c = 0; c < C; c++)
            for (int64_t q = 0; q < HW; q++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                out[o] = res[o] + mask[n] * gamma[c] * branch[o];
            }
}

/* Backward: gres = gy, gbranch = mask[n] * gamma[c] * gy,
 * ggamma[c] = sum over (n, q) of mask[n] * branch * gy. */
void or_layerscale_droppath_bwd(int N, int C, int64_t HW, const double* branch, const double* gamma,
                                const double* mask, const double* gy, double* gres, double* gbranch,
                                double* ggamma) {
    for (int c = 0; c < C; c++) ggamma[c] = 0.0;
    for (int n = 0; n < N; n++)
        for (int c = 0; c < C; c++)
            for (int64_t q = 0; q < HW; q++) {
                const int64_t o = ((int64_t)n * C + c) * HW + q;
                if (gres) gres[o] = gy[o];
                gbranch[o] = mask[n] * gamma[c] * gy[o];
                ggamma[c] += mask[n] * branch[o] * gy[o];
            }
}
