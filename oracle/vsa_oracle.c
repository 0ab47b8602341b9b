/*
 * vsa_oracle.c -- plain, slow CPU oracle for VSA (Video Sparse Attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; the two are compared against each other, and this file is
 * pinned on its own by the tests (brute force, closed forms, dense-attention
 * special cases, autograd and finite differences).
 *
 * Every quantity is float64 and every step is written as plain loops in the
 * order the method states it.  Tensors are contiguous [BH, N, d] (BH = batch
 * x heads, N tokens, d head dim); pooled tensors are [BH, Nc, d] with
 * Nc = N / 64.  OpenMP only splits independent rows across threads; it never
 * changes the order of any sum.
 *
 * Sources (cited by page and section):
 *  [AMD] "VSA: Accelerating Video Diffusion Inference with Sparse Attention on
 *        AMD GPUs" (ROCm blog).
 *  [ABS] "VSA: Faster Video Diffusion with Trainable Sparse Attention",
 *        Abstract.
 *
 * Readings where the pages are silent:
 *  - The 3D space-filling curve orders cubes of (4,4,4) tokens; tokens inside
 *    a cube stay in (t%4, h%4, w%4) raster order.  Two cube orders are
 *    provided: cube-raster order (t/4, h/4, w/4) -- the default -- and the
 *    3-D Hilbert curve of the enclosing power-of-two cube grid with the cells
 *    outside the grid skipped ("clipped" Hilbert order; the curve itself is
 *    J. Skilling's, "Programming the Hilbert curve", AIP Conf. Proc. 707,
 *    2004).  Every function taking `rank` uses rank[raster cube id] as the
 *    cube's position in the sequence; rank == NULL means raster order.
 *  - Coarse scores carry the SDPA scale (the pseudocode einsum in [AMD]
 *    "Generating Sparsity Patterns" shows none; Top-K is unaffected).
 *  - The coarse output is softmax(Sc) Vc over all cubes, broadcast to the
 *    64 tokens of each query cube.
 *  - The gated combination is out = g_c * O_c + g_f * O_f elementwise; a
 *    missing gate means all ones.
 *  - Top-K ties go to the lower cube id; the index list is stored in
 *    selection order (descending score), as torch.topk returns it.
 *  - A query cube with zero valid blocks has O_f = 0 and LSE = -inf.
 *  - A grid side that is not a multiple of 4 is covered by ceil(side / 4)
 *    cubes; a boundary cube keeps its 64 slots, and the slots whose token
 *    would lie outside the grid are padding: zero in the reordered tensors,
 *    left out of the cube's mean (which divides by the number of real
 *    tokens), never attended to as keys, and never written back.  The
 *    reordered length is Np = 64 * Nc >= N = T * H * W.
 *  - The Top-K set is a constant in the backward pass.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CUBE 64 /* (Ct, Ch, Cw) = (4, 4, 4) tokens per cube */

/* ------------------------------------------------------------------------ */
/* Pre-stage: 3D space-filling-curve token reordering.
 * [AMD] "Two-Stage Architecture", "Pre-stage: 3D Space-Filling Curve (SFC)
 * Token Reordering": tokens are remapped so that each fixed-size block of the
 * 1D sequence is a contiguous spatio-temporal region. */

/* Point x[0..2] (t, h, w) of the 3-D Hilbert curve of order b (a side of
 * 2^b cells) at curve index hidx, following Skilling's construction read
 * from index to point: the index's bits, taken three at a time from the
 * top, form the "transposed" coordinates (the first of each three bits goes
 * to t, the second to h, the third to w); these are Gray-decoded, and the
 * rotations and reflections the curve applies at each level are then undone
 * from the lowest level up. */
void orc_hilbert_point(uint64_t hidx, int b, uint32_t x[3])
{
    x[0] = x[1] = x[2] = 0;
    for (int level = b - 1; level >= 0; level--)
        for (int a = 0; a < 3; a++)
            x[a] |= (uint32_t)((hidx >> (3 * level + 2 - a)) & 1u) << level;
    if (b == 0)
        return;
    /* Gray decode: each axis takes the parity of the axes before it; the
     * first axis takes the last axis shifted down one level. */
    uint32_t carry = x[2] >> 1;
    x[2] ^= x[1];
    x[1] ^= x[0];
    x[0] ^= carry;
    /* Undo the per-level transforms, low level first. */
    for (uint32_t bit = 2; bit < (1u << b); bit <<= 1) {
        uint32_t low = bit - 1;
        for (int a = 2; a >= 0; a--) {
            if (x[a] & bit) {
                x[0] ^= low;               /* reflection of the low bits */
            } else {
                uint32_t swap = (x[0] ^ x[a]) & low;  /* exchange with axis 0 */
                x[0] ^= swap;
                x[a] ^= swap;
            }
        }
    }
}

/* rank[c] = position of raster cube c = (ct * Hc + ch) * Wc + cw in the cube
 * sequence.  curve 0: raster order (rank[c] = c).  curve 1: clipped Hilbert
 * order -- walk the Hilbert curve of the smallest 2^b >= max(Tc, Hc, Wc)
 * cube grid and number the cells that lie inside the grid in the order the
 * curve meets them. */
void orc_cube_rank(int Tc, int Hc, int Wc, int curve, int32_t *rank)
{
    const int64_t Nc = (int64_t)Tc * Hc * Wc;
    if (curve == 0) {
        for (int64_t c = 0; c < Nc; c++)
            rank[c] = (int32_t)c;
        return;
    }
    int b = 0;
    while ((1 << b) < Tc || (1 << b) < Hc || (1 << b) < Wc)
        b++;
    int32_t next = 0;
    for (uint64_t hidx = 0; hidx < ((uint64_t)1 << (3 * b)); hidx++) {
        uint32_t x[3];
        orc_hilbert_point(hidx, b, x);
        if (x[0] < (uint32_t)Tc && x[1] < (uint32_t)Hc && x[2] < (uint32_t)Wc)
            rank[((int64_t)x[0] * Hc + x[1]) * Wc + x[2]] = next++;
    }
}

/* Position in the reordered sequence of native token (t, h, w). */
int64_t orc_sfc_position(int t, int h, int w, int T, int H, int W, const int32_t *rank)
{
    (void)T;
    int64_t cube_t = t / 4, cube_h = h / 4, cube_w = w / 4;
    int64_t cubes_h = (H + 3) / 4, cubes_w = (W + 3) / 4;
    int64_t cube = (cube_t * cubes_h + cube_h) * cubes_w + cube_w;
    if (rank)
        cube = rank[cube];
    int64_t off = ((int64_t)(t % 4) * 4 + (h % 4)) * 4 + (w % 4);
    return cube * CUBE + off;
}

/* pos[n] = reordered position of the native token n = (t*H + h)*W + w. */
void orc_sfc_table(int T, int H, int W, const int32_t *rank, int64_t *pos)
{
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++)
            for (int w = 0; w < W; w++) {
                int64_t n = ((int64_t)t * H + h) * W + w;
                pos[n] = orc_sfc_position(t, h, w, T, H, W, rank);
            }
}

/* Number of cubes covering the grid, and the reordered length 64 * Nc. */
int64_t orc_num_cubes(int T, int H, int W)
{
    return (int64_t)((T + 3) / 4) * ((H + 3) / 4) * ((W + 3) / 4);
}

/* inverse == 0: y[pos[n]] = x[n] (native [BH, N, d] -> cube order
 * [BH, Np, d], padding slots zero); inverse != 0: y[n] = x[pos[n]] (cube
 * order -> native; padding slots are dropped). */
void orc_permute(const double *x, double *y, int64_t BH, int d,
                 int T, int H, int W, const int32_t *rank, int inverse)
{
    int64_t N = (int64_t)T * H * W, Np = CUBE * orc_num_cubes(T, H, W);
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * N);
    orc_sfc_table(T, H, W, rank, pos);
    if (!inverse)
        memset(y, 0, sizeof(double) * BH * Np * d);
#pragma omp parallel for
    for (int64_t bh = 0; bh < BH; bh++)
        for (int64_t n = 0; n < N; n++) {
            const double *src = inverse ? x + (bh * Np + pos[n]) * d : x + (bh * N + n) * d;
            double *dst = inverse ? y + (bh * N + n) * d : y + (bh * Np + pos[n]) * d;
            for (int c = 0; c < d; c++)
                dst[c] = src[c];
        }
    free(pos);
}

/* ------------------------------------------------------------------------ */
/* Stage 1: cube mean-pool.  [AMD] "Stage 1: Coarse Selection": each cube of
 * 64 tokens is mean-pooled into one cube-level vector (Qc, Kc, Vc).
 * Input is in reordered (cube-contiguous) order. */
/* ntok[c]: real tokens of cube c (NULL: 64 each); padding slots are zero,
 * so the sum over the 64 slots is the sum over the real tokens. */
void orc_pool(const double *xp, double *xc, int64_t BH, int64_t N, int d, const int32_t *ntok)
{
    int64_t Nc = N / CUBE;
#pragma omp parallel for
    for (int64_t bh = 0; bh < BH; bh++)
        for (int64_t c = 0; c < Nc; c++)
            for (int k = 0; k < d; k++) {
                double s = 0.0;
                for (int o = 0; o < CUBE; o++)
                    s += xp[(bh * N + c * CUBE + o) * d + k];
                xc[(bh * Nc + c) * d + k] = s / (ntok ? ntok[c] : CUBE);
            }
}

/* slot_ok[p] = 1 when reordered position p holds a token of the grid (0 for
 * padding), p in [0, Np); ntok[c] = number of tokens in cube position c. */
void orc_cube_slots(int T, int H, int W, const int32_t *rank, unsigned char *slot_ok, int32_t *ntok)
{
    int64_t N = (int64_t)T * H * W, Nc = orc_num_cubes(T, H, W);
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * N);
    orc_sfc_table(T, H, W, rank, pos);
    memset(slot_ok, 0, (size_t)(Nc * CUBE));
    for (int64_t c = 0; c < Nc; c++)
        ntok[c] = 0;
    for (int64_t n = 0; n < N; n++) {
        slot_ok[pos[n]] = 1;
        ntok[pos[n] / CUBE]++;
    }
    free(pos);
}

/* Stage 1: coarse cube-to-cube attention.
 * [AMD] "Stage 1: Coarse Selection" (cube-to-cube scores) and
 * "Stage 2: Fine Computation" (the coarse-stage output keeps global context);
 * the scale is the SDPA one of [AMD] "The Attention Bottleneck in Video
 * Diffusion".  scores [BH, Nc, Nc] (may be NULL), oc [BH, Nc, d] (may be
 * NULL), lse_c [BH, Nc] (may be NULL). */
void orc_coarse(const double *qc, const double *kc, const double *vc,
                int64_t BH, int Nc, int d, double scale,
                double *scores, double *oc, double *lse_c)
{
#pragma omp parallel for
    for (int64_t r = 0; r < BH * Nc; r++) {
        int64_t bh = r / Nc;
        double *s = (double *)malloc(sizeof(double) * Nc);
        const double *q = qc + r * d;
        for (int b = 0; b < Nc; b++) {
            const double *k = kc + (bh * Nc + b) * d;
            double dot = 0.0;
            for (int c = 0; c < d; c++)
                dot += q[c] * k[c];
            s[b] = scale * dot;
        }
        if (scores)
            for (int b = 0; b < Nc; b++)
                scores[r * Nc + b] = s[b];
        double m = -INFINITY;
        for (int b = 0; b < Nc; b++)
            if (s[b] > m)
                m = s[b];
        double l = 0.0;
        for (int b = 0; b < Nc; b++)
            l += exp(s[b] - m);
        if (lse_c)
            lse_c[r] = m + log(l);
        if (oc)
            for (int c = 0; c < d; c++) {
                double acc = 0.0;
                for (int b = 0; b < Nc; b++)
                    acc += exp(s[b] - m) / l * vc[(bh * Nc + b) * d + c];
                oc[r * d + c] = acc;
            }
        free(s);
    }
}

/* Stage 1: per-query-cube Top-K.  [AMD] "Stage 1: Coarse Selection" and the
 * torch.topk call in "Generating Sparsity Patterns": the K key cubes with the
 * highest scores, highest first; ties go to the lower cube id.
 * scores [rows, Nc] (rows = BH * number of query cubes); idx [rows, K]. */
typedef struct {
    double score;
    int32_t id;
} orc_scored_t;

static int orc_cmp_desc(const void *pa, const void *pb)
{
    const orc_scored_t *a = (const orc_scored_t *)pa;
    const orc_scored_t *b = (const orc_scored_t *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

void orc_topk(const double *scores, int64_t rows, int Nc, int K, int32_t *idx)
{
#pragma omp parallel for
    for (int64_t r = 0; r < rows; r++) {
        orc_scored_t *row = (orc_scored_t *)malloc(sizeof(orc_scored_t) * Nc);
        for (int b = 0; b < Nc; b++) {
            row[b].score = scores[r * Nc + b];
            row[b].id = b;
        }
        qsort(row, Nc, sizeof(orc_scored_t), orc_cmp_desc);
        for (int k = 0; k < K; k++)
            idx[r * K + k] = row[k].id;
        free(row);
    }
}

/* ------------------------------------------------------------------------ */
/* Stage 2: fine token-level attention over the selected cubes only.
 * [AMD] "Stage 2: Fine Computation" and "Sparse Traversal": for query block
 * q, visit kv_block_idx[q][i] for i < valid_block_num[q]; unselected cubes are
 * skipped.  The softmax is the SDPA one over the union of the selected cubes'
 * tokens.  One row: query token i (reordered order) of head bh. */
static void orc_fine_row(const double *qp, const double *kp, const double *vp,
                         const int32_t *idx, const int32_t *cnt, int Kmax,
                         int64_t N, int d, double scale, const unsigned char *slot_ok,
                         int64_t bh, int64_t i, double *of_row, double *lse_row)
{
    int64_t Nc = N / CUBE;
    int64_t qcube = i / CUBE;
    int n = cnt[bh * Nc + qcube];
    const int32_t *list = idx + (bh * Nc + qcube) * Kmax;
    const double *q = qp + (bh * N + i) * d;
    int64_t nk = (int64_t)n * CUBE;
    if (nk == 0) {
        for (int c = 0; c < d; c++)
            of_row[c] = 0.0;
        *lse_row = -INFINITY;
        return;
    }
    double *s = (double *)malloc(sizeof(double) * nk);
    for (int e = 0; e < n; e++)
        for (int o = 0; o < CUBE; o++) {
            int64_t j = (int64_t)list[e] * CUBE + o;
            const double *k = kp + (bh * N + j) * d;
            double dot = 0.0;
            for (int c = 0; c < d; c++)
                dot += q[c] * k[c];
            s[e * CUBE + o] = (slot_ok && !slot_ok[j]) ? -INFINITY : scale * dot;  /* padding: no key */
        }
    double m = -INFINITY;
    for (int64_t a = 0; a < nk; a++)
        if (s[a] > m)
            m = s[a];
    double l = 0.0;
    for (int64_t a = 0; a < nk; a++)
        l += exp(s[a] - m);
    *lse_row = m + log(l);
    for (int c = 0; c < d; c++) {
        double acc = 0.0;
        for (int e = 0; e < n; e++)
            for (int o = 0; o < CUBE; o++) {
                int64_t j = (int64_t)list[e] * CUBE + o;
                acc += exp(s[e * CUBE + o] - m) / l * vp[(bh * N + j) * d + c];
            }
        of_row[c] = acc;
    }
    free(s);
}

/* slot_ok (NULL: every slot holds a token) masks padding keys out. */
void orc_fine_fwd(const double *qp, const double *kp, const double *vp,
                  const int32_t *idx, const int32_t *cnt, int Kmax,
                  int64_t BH, int64_t N, int d, double scale,
                  const unsigned char *slot_ok, double *of, double *lse)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < BH * N; r++)
        orc_fine_row(qp, kp, vp, idx, cnt, Kmax, N, d, scale, slot_ok, r / N, r % N,
                     of + r * d, lse + r);
}

/* Same as orc_fine_fwd on a list of rows (r = bh*N + i), for sampled checks
 * at full size.  of_rows [nrows, d], lse_rows [nrows]. */
void orc_fine_fwd_rows(const double *qp, const double *kp, const double *vp,
                       const int32_t *idx, const int32_t *cnt, int Kmax,
                       int64_t BH, int64_t N, int d, double scale,
                       const unsigned char *slot_ok, const int64_t *rows, int64_t nrows,
                       double *of_rows, double *lse_rows)
{
    (void)BH;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t a = 0; a < nrows; a++)
        orc_fine_row(qp, kp, vp, idx, cnt, Kmax, N, d, scale, slot_ok, rows[a] / N,
                     rows[a] % N, of_rows + a * d, lse_rows + a);
}

/* Gated combination, in reordered order.  [AMD] "Stage 2: Fine Computation"
 * (the output combines the coarse and fine outputs through learnable gates)
 * and "Algorithmic Design".  gc / gf may be NULL (all ones). */
void orc_combine(const double *gc, const double *gf, const double *oc,
                 const double *of, int64_t BH, int64_t N, int d, double *outp)
{
    int64_t Nc = N / CUBE;
#pragma omp parallel for
    for (int64_t bh = 0; bh < BH; bh++)
        for (int64_t i = 0; i < N; i++)
            for (int c = 0; c < d; c++) {
                int64_t e = (bh * N + i) * d + c;
                double a = gc ? gc[e] : 1.0;
                double b = gf ? gf[e] : 1.0;
                outp[e] = a * oc[(bh * Nc + i / CUBE) * d + c] + b * of[e];
            }
}

void orc_lut_add_neighbors(const int32_t *idx_in, const int32_t *cnt_in, int kin, int64_t BH, int Tc, int Hc,
                           int Wc, const int32_t *rank, int radius, int kout, int32_t *idx_out, int32_t *cnt_out,
                           int *overflow);

/* The whole forward pass, native order in and out.
 * q, k, v, gc, gf: [BH, N, d] native (t, h, w) order; gc, gf may be NULL.
 * The selected key cubes of each query cube: lut_in, if not NULL ([BH, Nc,
 * kmax] lists with counts cnt_in, NULL meaning kmax for every query cube);
 * otherwise the Top-K of each coarse score row ([AMD] "Stage 1: Coarse
 * Selection"), united, when radius >= 0, with the cubes whose (t, h, w) cube
 * coordinates each differ from the query cube's by at most radius ([AMD]
 * "Comparison with Jenga": the block selection as the union of an importance
 * and an adjacency mask); the lists are then ascending, kmax wide (kmax = K
 * when radius < 0).
 * Outputs (all caller-allocated):
 *   out [BH, N, d] native; idx [BH, Nc, kmax]; cnt [BH, Nc]; of [BH, Np, d]
 *   and lse [BH, Np] (reordered order, Np = 64 Nc); oc [BH, Nc, d]; scores
 *   [BH, Nc, Nc] (may be NULL). */
void orc_forward(const double *q, const double *k, const double *v,
                 const double *gc, const double *gf, int64_t BH, int d,
                 int T, int H, int W, const int32_t *rank, int K, int radius, int kmax, double scale,
                 const int32_t *lut_in, const int32_t *cnt_in, double *out, int32_t *idx, int32_t *cnt,
                 double *of, double *lse, double *oc, double *scores)
{
    int64_t Nc = orc_num_cubes(T, H, W), N = Nc * CUBE;  /* N: reordered length */
    size_t big = sizeof(double) * BH * N * d, small = sizeof(double) * BH * Nc * d;
    unsigned char *slot_ok = (unsigned char *)malloc((size_t)N);
    int32_t *ntok = (int32_t *)malloc(sizeof(int32_t) * Nc);
    orc_cube_slots(T, H, W, rank, slot_ok, ntok);
    double *qp = (double *)malloc(big), *kp = (double *)malloc(big), *vp = (double *)malloc(big);
    double *qc = (double *)malloc(small), *kc = (double *)malloc(small), *vc = (double *)malloc(small);
    double *sc = scores ? scores : (double *)malloc(sizeof(double) * BH * Nc * Nc);
    orc_permute(q, qp, BH, d, T, H, W, rank, 0);
    orc_permute(k, kp, BH, d, T, H, W, rank, 0);
    orc_permute(v, vp, BH, d, T, H, W, rank, 0);
    orc_pool(qp, qc, BH, N, d, ntok);
    orc_pool(kp, kc, BH, N, d, ntok);
    orc_pool(vp, vc, BH, N, d, ntok);
    orc_coarse(qc, kc, vc, BH, (int)Nc, d, scale, sc, oc, NULL);
    if (lut_in) {
        memcpy(idx, lut_in, sizeof(int32_t) * BH * Nc * kmax);
        for (int64_t r = 0; r < BH * Nc; r++)
            cnt[r] = cnt_in ? cnt_in[r] : kmax;
    } else if (radius < 0) {
        orc_topk(sc, BH * Nc, (int)Nc, K, idx);
        for (int64_t r = 0; r < BH * Nc; r++)
            cnt[r] = K;
    } else {
        int32_t *tk = (int32_t *)malloc(sizeof(int32_t) * BH * Nc * K);
        int overflow = 0;
        orc_topk(sc, BH * Nc, (int)Nc, K, tk);
        orc_lut_add_neighbors(tk, NULL, K, BH, (T + 3) / 4, (H + 3) / 4, (W + 3) / 4, rank, radius, kmax, idx, cnt,
                              &overflow);
        free(tk);
    }
    orc_fine_fwd(qp, kp, vp, idx, cnt, kmax, BH, N, d, scale, slot_ok, of, lse);
    double *gcp = NULL, *gfp = NULL, *outp = (double *)malloc(big);
    if (gc) {
        gcp = (double *)malloc(big);
        orc_permute(gc, gcp, BH, d, T, H, W, rank, 0);
    }
    if (gf) {
        gfp = (double *)malloc(big);
        orc_permute(gf, gfp, BH, d, T, H, W, rank, 0);
    }
    orc_combine(gcp, gfp, oc, of, BH, N, d, outp);
    orc_permute(outp, out, BH, d, T, H, W, rank, 1);
    free(qp); free(kp); free(vp); free(qc); free(kc); free(vc);
    if (!scores) free(sc);
    free(gcp); free(gfp); free(outp); free(slot_ok); free(ntok);
}

/* ------------------------------------------------------------------------ */
/* Backward.  [ABS]: VSA trains end to end as one differentiable operator.
 * The derivative of each step is the textbook one (softmax Jacobian
 * dS = P * (dP - sum_k P dP)); the Top-K selection is held constant. */

/* Fine stage backward, reordered order.  dof = dL/dO_f.  dq, dk, dv are
 * overwritten. */
void orc_fine_bwd(const double *qp, const double *kp, const double *vp,
                  const double *dof, const int32_t *idx, const int32_t *cnt,
                  int Kmax, int64_t BH, int64_t N, int d, double scale,
                  const unsigned char *slot_ok, double *dq, double *dk, double *dv)
{
    int64_t Nc = N / CUBE;
    memset(dq, 0, sizeof(double) * BH * N * d);
    memset(dk, 0, sizeof(double) * BH * N * d);
    memset(dv, 0, sizeof(double) * BH * N * d);
    /* Heads are independent; inside a head the rows are visited in order. */
#pragma omp parallel for
    for (int64_t bh = 0; bh < BH; bh++) {
        int64_t maxk = (int64_t)Kmax * CUBE;
        double *s = (double *)malloc(sizeof(double) * (maxk + 1));
        double *p = (double *)malloc(sizeof(double) * (maxk + 1));
        double *dp = (double *)malloc(sizeof(double) * (maxk + 1));
        int64_t *key = (int64_t *)malloc(sizeof(int64_t) * (maxk + 1));
        for (int64_t i = 0; i < N; i++) {
            int64_t qcube = i / CUBE;
            int n = cnt[bh * Nc + qcube];
            const int32_t *list = idx + (bh * Nc + qcube) * Kmax;
            int64_t nk = (int64_t)n * CUBE;
            if (nk == 0)
                continue;
            const double *q = qp + (bh * N + i) * d;
            const double *g = dof + (bh * N + i) * d;
            for (int e = 0; e < n; e++)
                for (int o = 0; o < CUBE; o++)
                    key[e * CUBE + o] = (int64_t)list[e] * CUBE + o;
            double m = -INFINITY;
            for (int64_t a = 0; a < nk; a++) {
                const double *kk = kp + (bh * N + key[a]) * d;
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += q[c] * kk[c];
                s[a] = (slot_ok && !slot_ok[key[a]]) ? -INFINITY : scale * dot;
                if (s[a] > m)
                    m = s[a];
            }
            double l = 0.0;
            for (int64_t a = 0; a < nk; a++)
                l += exp(s[a] - m);
            for (int64_t a = 0; a < nk; a++)
                p[a] = exp(s[a] - m) / l;
            /* dP_ij = dO_i . V_j ; D_i = sum_j P_ij dP_ij */
            double D = 0.0;
            for (int64_t a = 0; a < nk; a++) {
                const double *vv = vp + (bh * N + key[a]) * d;
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += g[c] * vv[c];
                dp[a] = dot;
                D += p[a] * dot;
            }
            double *dqi = dq + (bh * N + i) * d;
            for (int64_t a = 0; a < nk; a++) {
                double ds = p[a] * (dp[a] - D);
                const double *kk = kp + (bh * N + key[a]) * d;
                double *dkj = dk + (bh * N + key[a]) * d;
                double *dvj = dv + (bh * N + key[a]) * d;
                for (int c = 0; c < d; c++) {
                    dvj[c] += p[a] * g[c];
                    dqi[c] += scale * ds * kk[c];
                    dkj[c] += scale * ds * q[c];
                }
            }
        }
        free(s); free(p); free(dp); free(key);
    }
}

/* Sampled fine backward, for checks at full size.
 * dQ of the listed query rows r = bh*N + i (dq_rows [nrows, d]); the row's
 * softmax, dP and D are recomputed from scratch exactly as orc_fine_bwd does. */
void orc_fine_bwd_query_rows(const double *qp, const double *kp, const double *vp,
                             const double *dof, const int32_t *idx, const int32_t *cnt,
                             int Kmax, int64_t N, int d, double scale, const unsigned char *slot_ok,
                             const int64_t *rows, int64_t nrows, double *dq_rows)
{
    int64_t Nc = N / CUBE;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t a = 0; a < nrows; a++) {
        int64_t bh = rows[a] / N, i = rows[a] % N;
        int64_t qcube = i / CUBE;
        int n = cnt[bh * Nc + qcube];
        const int32_t *list = idx + (bh * Nc + qcube) * Kmax;
        int64_t nk = (int64_t)n * CUBE;
        double *out = dq_rows + a * d;
        for (int c = 0; c < d; c++)
            out[c] = 0.0;
        if (nk == 0)
            continue;
        double *s = (double *)malloc(sizeof(double) * nk);
        double *dp = (double *)malloc(sizeof(double) * nk);
        const double *q = qp + (bh * N + i) * d;
        const double *g = dof + (bh * N + i) * d;
        double m = -INFINITY;
        for (int64_t e = 0; e < nk; e++) {
            int64_t j = (int64_t)list[e / CUBE] * CUBE + e % CUBE;
            const double *kk = kp + (bh * N + j) * d;
            const double *vv = vp + (bh * N + j) * d;
            double dot = 0.0, dot2 = 0.0;
            for (int c = 0; c < d; c++) {
                dot += q[c] * kk[c];
                dot2 += g[c] * vv[c];
            }
            s[e] = (slot_ok && !slot_ok[j]) ? -INFINITY : scale * dot;
            dp[e] = dot2;
            if (s[e] > m)
                m = s[e];
        }
        double l = 0.0;
        for (int64_t e = 0; e < nk; e++)
            l += exp(s[e] - m);
        double D = 0.0;
        for (int64_t e = 0; e < nk; e++)
            D += exp(s[e] - m) / l * dp[e];
        for (int64_t e = 0; e < nk; e++) {
            double ds = exp(s[e] - m) / l * (dp[e] - D);
            int64_t j = (int64_t)list[e / CUBE] * CUBE + e % CUBE;
            const double *kk = kp + (bh * N + j) * d;
            for (int c = 0; c < d; c++)
                out[c] += scale * ds * kk[c];
        }
        free(s);
        free(dp);
    }
}

/* dK and dV of the 64 tokens of key cube `kcube` of head bh: the sum over
 * every query row whose cube lists kcube.  dk_rows, dv_rows [64, d]. */
void orc_fine_bwd_key_cube(const double *qp, const double *kp, const double *vp,
                           const double *dof, const int32_t *idx, const int32_t *cnt,
                           int Kmax, int64_t N, int d, double scale, const unsigned char *slot_ok,
                           int64_t bh, int kcube, double *dk_rows, double *dv_rows)
{
    int64_t Nc = N / CUBE;
    for (int64_t e = 0; e < (int64_t)CUBE * d; e++) {
        dk_rows[e] = 0.0;
        dv_rows[e] = 0.0;
    }
    int64_t maxk = (int64_t)Kmax * CUBE;
    /* Query rows are independent; each thread sums its rows' contributions
     * and the partial sums are added at the end (only the order of the
     * additions depends on the thread count). */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (maxk + 1));
        double *dp = (double *)malloc(sizeof(double) * (maxk + 1));
        double *dk_part = (double *)calloc((size_t)CUBE * d, sizeof(double));
        double *dv_part = (double *)calloc((size_t)CUBE * d, sizeof(double));
#pragma omp for schedule(dynamic, 64)
        for (int64_t i = 0; i < N; i++) {
            int64_t qcube = i / CUBE;
            int n = cnt[bh * Nc + qcube];
            const int32_t *list = idx + (bh * Nc + qcube) * Kmax;
            int hit = -1;
            for (int e = 0; e < n; e++)
                if (list[e] == kcube)
                    hit = e;
            if (hit < 0)
                continue;
            int64_t nk = (int64_t)n * CUBE;
            const double *q = qp + (bh * N + i) * d;
            const double *g = dof + (bh * N + i) * d;
            double m = -INFINITY;
            for (int64_t e = 0; e < nk; e++) {
                int64_t j = (int64_t)list[e / CUBE] * CUBE + e % CUBE;
                const double *kk = kp + (bh * N + j) * d;
                const double *vv = vp + (bh * N + j) * d;
                double dot = 0.0, dot2 = 0.0;
                for (int c = 0; c < d; c++) {
                    dot += q[c] * kk[c];
                    dot2 += g[c] * vv[c];
                }
                s[e] = (slot_ok && !slot_ok[j]) ? -INFINITY : scale * dot;
                dp[e] = dot2;
                if (s[e] > m)
                    m = s[e];
            }
            double l = 0.0;
            for (int64_t e = 0; e < nk; e++)
                l += exp(s[e] - m);
            double D = 0.0;
            for (int64_t e = 0; e < nk; e++)
                D += exp(s[e] - m) / l * dp[e];
            for (int o = 0; o < CUBE; o++) {
                int64_t e = (int64_t)hit * CUBE + o;
                double p = exp(s[e] - m) / l;
                double ds = p * (dp[e] - D);
                for (int c = 0; c < d; c++) {
                    dv_part[o * d + c] += p * g[c];
                    dk_part[o * d + c] += scale * ds * q[c];
                }
            }
        }
#pragma omp critical
        for (int64_t e = 0; e < (int64_t)CUBE * d; e++) {
            dk_rows[e] += dk_part[e];
            dv_rows[e] += dv_part[e];
        }
        free(s);
        free(dp);
        free(dk_part);
        free(dv_part);
    }
}

/* Backward of the gated combination, reordered order: dout_p = dL/dout.
 * dof = g_f * dO; doc[cube] = sum over the cube of g_c * dO; dgc = dO * O_c;
 * dgf = dO * O_f.  gc / gf may be NULL (ones). */
void orc_combine_bwd(const double *dout_p, const double *gc, const double *gf,
                     const double *oc, const double *of, int64_t BH, int64_t N, int d,
                     double *dof, double *doc, double *dgc, double *dgf)
{
    int64_t Nc = N / CUBE;
    memset(doc, 0, sizeof(double) * BH * Nc * d);
    for (int64_t bh = 0; bh < BH; bh++)
        for (int64_t i = 0; i < N; i++)
            for (int c = 0; c < d; c++) {
                int64_t e = (bh * N + i) * d + c;
                int64_t ec = (bh * Nc + i / CUBE) * d + c;
                double a = gc ? gc[e] : 1.0, b = gf ? gf[e] : 1.0;
                dof[e] = b * dout_p[e];
                doc[ec] += a * dout_p[e];
                dgc[e] = dout_p[e] * oc[ec];
                dgf[e] = dout_p[e] * of[e];
            }
}

/* Coarse stage backward: doc = dL/dO_c [BH, Nc, d]; outputs overwritten. */
void orc_coarse_bwd(const double *qc, const double *kc, const double *vc,
                    const double *doc, int64_t BH, int Nc, int d, double scale,
                    double *dqc, double *dkc, double *dvc)
{
    memset(dqc, 0, sizeof(double) * BH * Nc * d);
    memset(dkc, 0, sizeof(double) * BH * Nc * d);
    memset(dvc, 0, sizeof(double) * BH * Nc * d);
#pragma omp parallel for
    for (int64_t bh = 0; bh < BH; bh++) {
        double *s = (double *)malloc(sizeof(double) * Nc);
        double *p = (double *)malloc(sizeof(double) * Nc);
        double *dp = (double *)malloc(sizeof(double) * Nc);
        for (int a = 0; a < Nc; a++) {
            const double *q = qc + (bh * Nc + a) * d;
            const double *g = doc + (bh * Nc + a) * d;
            double m = -INFINITY;
            for (int b = 0; b < Nc; b++) {
                const double *k = kc + (bh * Nc + b) * d;
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += q[c] * k[c];
                s[b] = scale * dot;
                if (s[b] > m)
                    m = s[b];
            }
            double l = 0.0;
            for (int b = 0; b < Nc; b++)
                l += exp(s[b] - m);
            double D = 0.0;
            for (int b = 0; b < Nc; b++) {
                p[b] = exp(s[b] - m) / l;
                const double *v = vc + (bh * Nc + b) * d;
                double dot = 0.0;
                for (int c = 0; c < d; c++)
                    dot += g[c] * v[c];
                dp[b] = dot;
                D += p[b] * dot;
            }
            for (int b = 0; b < Nc; b++) {
                double ds = p[b] * (dp[b] - D);
                const double *k = kc + (bh * Nc + b) * d;
                for (int c = 0; c < d; c++) {
                    dvc[(bh * Nc + b) * d + c] += p[b] * g[c];
                    dqc[(bh * Nc + a) * d + c] += scale * ds * k[c];
                    dkc[(bh * Nc + b) * d + c] += scale * ds * q[c];
                }
            }
        }
        free(s); free(p); free(dp);
    }
}

/* The whole backward pass, native order in and out.
 * Inputs as orc_forward, plus the lists the forward used (idx [BH, Nc, kmax]
 * with counts cnt_in, NULL meaning kmax for every query cube) and dout
 * [BH, N, d] native.  Outputs (caller-allocated, native order): dq, dk, dv
 * [BH, N, d]; dgc, dgf [BH, N, d] (ignored when the gate is NULL). */
void orc_backward(const double *q, const double *k, const double *v,
                  const double *gc, const double *gf, int64_t BH, int d,
                  int T, int H, int W, const int32_t *rank, int kmax, double scale, const int32_t *idx,
                  const int32_t *cnt_in, const double *dout, double *dq, double *dk, double *dv,
                  double *dgc, double *dgf)
{
    int64_t Nc = orc_num_cubes(T, H, W), N = Nc * CUBE;  /* N: reordered length */
    size_t big = sizeof(double) * BH * N * d, small = sizeof(double) * BH * Nc * d;
    unsigned char *slot_ok = (unsigned char *)malloc((size_t)N);
    int32_t *ntok = (int32_t *)malloc(sizeof(int32_t) * Nc);
    orc_cube_slots(T, H, W, rank, slot_ok, ntok);
    double *qp = (double *)malloc(big), *kp = (double *)malloc(big), *vp = (double *)malloc(big);
    double *qc = (double *)malloc(small), *kc = (double *)malloc(small), *vc = (double *)malloc(small);
    double *oc = (double *)malloc(small), *of = (double *)malloc(big);
    double *lse = (double *)malloc(sizeof(double) * BH * N);
    double *dop = (double *)malloc(big), *gcp = (double *)malloc(big), *gfp = (double *)malloc(big);
    double *dgcp = (double *)malloc(big), *dgfp = (double *)malloc(big);
    double *dof = (double *)malloc(big), *doc = (double *)malloc(small);
    double *dqp = (double *)malloc(big), *dkp = (double *)malloc(big), *dvp = (double *)malloc(big);
    double *dqc = (double *)malloc(small), *dkc = (double *)malloc(small), *dvc = (double *)malloc(small);
    int32_t *cnt = (int32_t *)malloc(sizeof(int32_t) * BH * Nc);
    for (int64_t r = 0; r < BH * Nc; r++)
        cnt[r] = cnt_in ? cnt_in[r] : kmax;

    /* Recompute the forward intermediates. */
    orc_permute(q, qp, BH, d, T, H, W, rank, 0);
    orc_permute(k, kp, BH, d, T, H, W, rank, 0);
    orc_permute(v, vp, BH, d, T, H, W, rank, 0);
    orc_pool(qp, qc, BH, N, d, ntok);
    orc_pool(kp, kc, BH, N, d, ntok);
    orc_pool(vp, vc, BH, N, d, ntok);
    orc_coarse(qc, kc, vc, BH, (int)Nc, d, scale, NULL, oc, NULL);
    orc_fine_fwd(qp, kp, vp, idx, cnt, kmax, BH, N, d, scale, slot_ok, of, lse);

    /* Gated combination out_p = gc*Oc[cube] + gf*Of, differentiated. */
    orc_permute(dout, dop, BH, d, T, H, W, rank, 0);
    if (gc)
        orc_permute(gc, gcp, BH, d, T, H, W, rank, 0);
    if (gf)
        orc_permute(gf, gfp, BH, d, T, H, W, rank, 0);
    orc_combine_bwd(dop, gc ? gcp : NULL, gf ? gfp : NULL, oc, of, BH, N, d, dof, doc, dgcp, dgfp);
    if (gc && dgc)
        orc_permute(dgcp, dgc, BH, d, T, H, W, rank, 1);
    if (gf && dgf)
        orc_permute(dgfp, dgf, BH, d, T, H, W, rank, 1);

    orc_fine_bwd(qp, kp, vp, dof, idx, cnt, kmax, BH, N, d, scale, slot_ok, dqp, dkp, dvp);
    orc_coarse_bwd(qc, kc, vc, doc, BH, (int)Nc, d, scale, dqc, dkc, dvc);

    /* Mean-pool backward: every token of a cube gets dXc / (tokens in the
     * cube); padding slots are dropped by the inverse reordering. */
    for (int64_t bh = 0; bh < BH; bh++)
        for (int64_t i = 0; i < N; i++)
            for (int c = 0; c < d; c++) {
                int64_t e = (bh * N + i) * d + c, ec = (bh * Nc + i / CUBE) * d + c;
                dqp[e] += dqc[ec] / ntok[i / CUBE];
                dkp[e] += dkc[ec] / ntok[i / CUBE];
                dvp[e] += dvc[ec] / ntok[i / CUBE];
            }
    orc_permute(dqp, dq, BH, d, T, H, W, rank, 1);
    orc_permute(dkp, dk, BH, d, T, H, W, rank, 1);
    orc_permute(dvp, dv, BH, d, T, H, W, rank, 1);

    free(qp); free(kp); free(vp); free(qc); free(kc); free(vc); free(oc); free(of);
    free(lse); free(dop); free(gcp); free(gfp); free(dgcp); free(dgfp); free(dof); free(doc);
    free(dqp); free(dkp); free(dvp); free(dqc); free(dkc); free(dvc); free(cnt);
    free(slot_ok); free(ntok);
}

/* ---- index-list conversions ("Sparse Encoding in CK Tile": Jenga's M x M
 * block matrix B vs VSA's selected-block list plus valid count; "Comparison
 * with Jenga", "Algorithmic Design": adjacency as one of Jenga's masks). */

/* Row r of a keep-set (sel[0..Nc)) as an ascending list of at most kmax ids,
 * -1 after the count; a longer row keeps its lowest ids and sets *overflow. */
static void orc_write_list(const unsigned char *sel, int Nc, int kmax, int32_t *idx, int32_t *cnt, int *overflow)
{
    int n = 0;
    for (int j = 0; j < Nc; j++) {
        if (!sel[j])
            continue;
        if (n < kmax)
            idx[n] = j;
        n++;
    }
    if (n > kmax) {
        *overflow = 1;
        n = kmax;
    }
    for (int e = n; e < kmax; e++)
        idx[e] = -1;
    *cnt = n;
}

/* mask[row][j] != 0: query cube `row % Nc` keeps key cube j. */
void orc_mask_to_lut(const unsigned char *mask, int64_t rows, int Nc, int kmax, int32_t *idx, int32_t *cnt,
                     int *overflow)
{
    *overflow = 0;
    for (int64_t r = 0; r < rows; r++)
        orc_write_list(mask + r * Nc, Nc, kmax, idx + r * kmax, cnt + r, overflow);
}

/* The list of every query cube united with all cubes whose cube-grid
 * coordinates (t, h, w) each differ from the query cube's by at most
 * `radius`.  Cube ids are positions in the cube sequence: raster cube
 * (t * Hc + h) * Wc + w sits at position rank[raster id] (rank NULL: the
 * raster id itself). */
void orc_lut_add_neighbors(const int32_t *idx_in, const int32_t *cnt_in, int kin, int64_t BH, int Tc, int Hc,
                           int Wc, const int32_t *rank, int radius, int kout, int32_t *idx_out, int32_t *cnt_out,
                           int *overflow)
{
    const int Nc = Tc * Hc * Wc;
    *overflow = 0;
    unsigned char *sel = (unsigned char *)malloc((size_t)Nc);
    int *raster_of = (int *)malloc(sizeof(int) * (size_t)Nc);  /* position -> raster id */
    for (int r = 0; r < Nc; r++)
        raster_of[rank ? rank[r] : r] = r;
    for (int64_t bh = 0; bh < BH; bh++) {
        for (int q = 0; q < Nc; q++) {
            const int64_t row = bh * Nc + q;
            memset(sel, 0, (size_t)Nc);
            int n = cnt_in ? cnt_in[row] : kin;
            if (n < 0)
                n = 0;
            if (n > kin)
                n = kin;
            for (int e = 0; e < n; e++) {
                int c = idx_in[row * kin + e];
                if (c >= 0 && c < Nc)
                    sel[c] = 1;
            }
            const int qr = raster_of[q];
            const int qt = qr / (Hc * Wc), qh = (qr / Wc) % Hc, qw = qr % Wc;
            for (int c = 0; c < Nc; c++) {
                const int cr = raster_of[c];
                const int t = cr / (Hc * Wc), h = (cr / Wc) % Hc, w = cr % Wc;
                if (abs(t - qt) <= radius && abs(h - qh) <= radius && abs(w - qw) <= radius)
                    sel[c] = 1;
            }
            orc_write_list(sel, Nc, kout, idx_out + row * kout, cnt_out + row, overflow);
        }
    }
    free(sel);
    free(raster_of);
}
