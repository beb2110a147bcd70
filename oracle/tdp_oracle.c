/*
 * tdp_oracle.c -- plain, slow CPU definition of the Tiled Data Parallelism (TDP)
 * tile split / position normalisation / conditioning filter / trapezoidal
 * blend.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the library itself never does.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Source: "Tiled Data Parallelism (TDP)" (LTX-2 docs, multigpu), sections
 * "What it is", "Position normalization", "Shared negative (reference)
 * positions" and "API / Tiling config".  Where the page leaves a step open,
 * the reading taken is stated beside the function that takes it.
 *
 * Conventions (all arrays contiguous, row-major, host memory):
 *   X     [B,F,H,W,C]          latent; elements of `esize` bytes (4 = fp32, 2 = bf16 bits)
 *   P     [B,3,T,2]  int32     generated-token [start,end) per dimension (F,H,W), T = F*H*W
 *   tiles t = (iF*nH + iH)*nW + iW, token order inside a tile row-major (f,h,w)
 *   Y     tile-major: tile t is a contiguous [B,T_t,C] block starting at token B*off_t
 *   Q     tile-major: tile t is a contiguous [B,3,T_t,2] int32 block
 *   mn,mx [nt,B,3]   int32     min start / max end of the tile's generated tokens
 *   K     [B,3,N,2]  int32     conditioning-token intervals
 *   keep  [nt,B,N]   uint8;  idx [nt,B,N] int32;  count [nt,B];  kcount [B,N];
 *   Kout  [nt,B,3,N,2] int32  kept tokens of (t,b), compacted in ascending k
 *   Z     [B,F,H,W,C] double   blended latent
 *
 * Position arithmetic wraps modulo 2^32 (two's complement), as int32 does on
 * the GPU; it is done through uint32 here to stay defined in C.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t B, F, H, W, C;
    int32_t esize;     /* bytes per latent element: 4 (fp32) or 2 (bf16 bit pattern) */
    int32_t n[3];      /* tiles per dimension (F, H, W) */
    int32_t o[3];      /* overlap per dimension, latent grid units */
} oracle_problem;

/* ------------------------------------------------------------------------
 * Tile boxes along one dimension ("API / Tiling config": a tile COUNT and an
 * overlap per dimension, not sizes; the box formula is not on the page).
 *
 * Reading taken: balanced cores c_i = floor(i*L/n), i = 0..n; tile i spans
 * [c_i - a, c_{i+1} + b) with a = floor(o/2), b = o - a, and no extension at
 * the outer edges.  Neighbours then overlap by exactly o.  Valid when n >= 1,
 * n <= L, o >= 0 and, for n >= 2, every core is at least o long (so that no
 * cell lies in two overlaps).  With n = 1 the overlap is ignored.
 * Returns 0, or -1 for an invalid (L, n, o).
 * ---------------------------------------------------------------------- */
int oracle_tile_boxes_1d(int32_t L, int32_t n, int32_t o, int32_t *lo, int32_t *hi)
{
    if (L < 1 || n < 1 || n > L || o < 0) return -1;
    if (n == 1) { lo[0] = 0; hi[0] = L; return 0; }
    int32_t a = o / 2, b = o - a;
    for (int32_t i = 0; i < n; ++i) {
        int32_t c0 = (int32_t)(((int64_t)i * L) / n);
        int32_t c1 = (int32_t)(((int64_t)(i + 1) * L) / n);
        if (c1 - c0 < o) return -1;
        lo[i] = (i > 0) ? c0 - a : c0;
        hi[i] = (i < n - 1) ? c1 + b : c1;
    }
    return 0;
}

static int32_t dim_len(const oracle_problem *p, int d)
{
    return d == 0 ? p->F : (d == 1 ? p->H : p->W);
}

int oracle_num_tiles(const oracle_problem *p)
{
    return p->n[0] * p->n[1] * p->n[2];
}

/* box[t][d][0..1] = [lo, hi) of tile t; off[t] = sum of T_u over u < t; off[nt] = total.
 * Returns 0, or -1 for invalid geometry. */
int oracle_plan(const oracle_problem *p, int32_t *box, int64_t *off)
{
    int32_t lo[3][4096], hi[3][4096];
    for (int d = 0; d < 3; ++d) {
        if (p->n[d] > 4096) return -1;
        if (oracle_tile_boxes_1d(dim_len(p, d), p->n[d], p->o[d], lo[d], hi[d]) != 0) return -1;
    }
    int nt = oracle_num_tiles(p);
    int64_t acc = 0;
    for (int t = 0; t < nt; ++t) {
        int i[3];
        i[0] = t / (p->n[1] * p->n[2]);
        i[1] = (t / p->n[2]) % p->n[1];
        i[2] = t % p->n[2];
        int64_t tt = 1;
        for (int d = 0; d < 3; ++d) {
            box[(t * 3 + d) * 2 + 0] = lo[d][i[d]];
            box[(t * 3 + d) * 2 + 1] = hi[d][i[d]];
            tt *= (int64_t)(hi[d][i[d]] - lo[d][i[d]]);
        }
        off[t] = acc;
        acc += tt;
    }
    off[nt] = acc;
    return 0;
}

/* ------------------------------------------------------------------------
 * Trapezoidal ramp ("What it is": overlaps are blended with trapezoidal
 * masks that sum to one everywhere; the ramp is not printed).
 *
 * Reading taken: inside the o-cell overlap of tiles i and i+1, with k = 0..o-1
 * counted from the overlap's left edge, tile i+1 weighs (k+1)/(o+1) and tile i
 * weighs (o-k)/(o+1); a tile weighs 1 elsewhere inside its box and 0 outside.
 * Returned as the integer numerator over the denominator o+1 (o taken as 0
 * when n = 1).
 * ---------------------------------------------------------------------- */
int32_t oracle_ramp_num(int32_t L, int32_t n, int32_t o, int32_t i, int32_t x, int32_t *den)
{
    int32_t lo[4096], hi[4096];
    if (n == 1) o = 0;
    *den = o + 1;
    if (n > 4096 || oracle_tile_boxes_1d(L, n, o, lo, hi) != 0) return -1;
    if (i < 0 || i >= n || x < lo[i] || x >= hi[i]) return 0;
    if (i > 0 && x < hi[i - 1]) return (x - lo[i]) + 1;           /* rising edge, shared with i-1 */
    if (i < n - 1 && x >= lo[i + 1]) return o - (x - lo[i + 1]);  /* falling edge, shared with i+1 */
    return o + 1;
}

static double ramp(const oracle_problem *p, int d, int32_t i, int32_t x)
{
    int32_t den;
    int32_t num = oracle_ramp_num(dim_len(p, d), p->n[d], p->o[d], i, x, &den);
    return (double)num / (double)den;
}

/* Separable 3-D mask of tile t at global cell (f,h,w), fp64: (r_F * r_H) * r_W. */
double oracle_mask(const oracle_problem *p, int32_t t, int32_t f, int32_t h, int32_t w)
{
    int32_t iF = t / (p->n[1] * p->n[2]);
    int32_t iH = (t / p->n[2]) % p->n[1];
    int32_t iW = t % p->n[2];
    return (ramp(p, 0, iF, f) * ramp(p, 1, iH, h)) * ramp(p, 2, iW, w);
}

/* ------------------------------------------------------------------------
 * tile_split ("What it is": the patchified (frames, height, width) latent is
 * split into tiles; each tile's tokens, with their positions, go to one
 * transformer call).  Plain copy of every token of every tile box.
 * ---------------------------------------------------------------------- */
void oracle_split(const oracle_problem *p, const void *X, const int32_t *P, void *Y, int32_t *Q)
{
    int nt = oracle_num_tiles(p);
    int32_t *box = (int32_t *)malloc(sizeof(int32_t) * 6 * (size_t)nt);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)nt + 1));
    oracle_plan(p, box, off);
    const int64_t T = (int64_t)p->F * p->H * p->W;
    const size_t row = (size_t)p->C * (size_t)p->esize;
    for (int t = 0; t < nt; ++t) {
        const int32_t *bx = box + t * 6;
        int64_t Tt = off[t + 1] - off[t];
        for (int32_t b = 0; b < p->B; ++b) {
            int64_t j = 0;
            for (int32_t f = bx[0]; f < bx[1]; ++f)
                for (int32_t h = bx[2]; h < bx[3]; ++h)
                    for (int32_t w = bx[4]; w < bx[5]; ++w, ++j) {
                        int64_t g = ((int64_t)f * p->H + h) * p->W + w;
                        const char *src = (const char *)X + ((int64_t)b * T + g) * (int64_t)row;
                        char *dst = (char *)Y + ((int64_t)p->B * off[t] + (int64_t)b * Tt + j) * (int64_t)row;
                        memcpy(dst, src, row);
                        for (int d = 0; d < 3; ++d)
                            for (int s = 0; s < 2; ++s)
                                Q[(((int64_t)p->B * off[t]) * 3 + ((int64_t)b * 3 + d) * Tt + j) * 2 + s] =
                                    P[(((int64_t)b * 3 + d) * T + g) * 2 + s];
                    }
        }
    }
    free(box);
    free(off);
}

/* ------------------------------------------------------------------------
 * Position bounds ("Position normalization": the offset is the minimum start
 * over the tile's generated tokens, per batch item and per dimension).
 * mx (maximum end) is the tile's far edge in position space, used by the
 * conditioning filter below.
 * ---------------------------------------------------------------------- */
void oracle_bounds(const oracle_problem *p, const int32_t *Q, int32_t *mn, int32_t *mx)
{
    int nt = oracle_num_tiles(p);
    int32_t *box = (int32_t *)malloc(sizeof(int32_t) * 6 * (size_t)nt);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)nt + 1));
    oracle_plan(p, box, off);
    for (int t = 0; t < nt; ++t) {
        int64_t Tt = off[t + 1] - off[t];
        for (int32_t b = 0; b < p->B; ++b)
            for (int d = 0; d < 3; ++d) {
                const int32_t *q = Q + (((int64_t)p->B * off[t]) * 3 + ((int64_t)b * 3 + d) * Tt) * 2;
                int32_t lo = q[0], hi = q[1];
                for (int64_t j = 1; j < Tt; ++j) {
                    if (q[2 * j] < lo) lo = q[2 * j];
                    if (q[2 * j + 1] > hi) hi = q[2 * j + 1];
                }
                mn[((int64_t)t * p->B + b) * 3 + d] = lo;
                mx[((int64_t)t * p->B + b) * 3 + d] = hi;
            }
    }
    free(box);
    free(off);
}

static int32_t wrap_sub(int32_t a, int32_t b)
{
    return (int32_t)((uint32_t)a - (uint32_t)b);
}

/* "Position normalization": positions -= offset, start and end alike, for
 * every generated token of the tile (widths are kept). */
void oracle_normalize(const oracle_problem *p, int32_t *Q, const int32_t *mn)
{
    int nt = oracle_num_tiles(p);
    int32_t *box = (int32_t *)malloc(sizeof(int32_t) * 6 * (size_t)nt);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)nt + 1));
    oracle_plan(p, box, off);
    for (int t = 0; t < nt; ++t) {
        int64_t Tt = off[t + 1] - off[t];
        for (int32_t b = 0; b < p->B; ++b)
            for (int d = 0; d < 3; ++d) {
                int32_t *q = Q + (((int64_t)p->B * off[t]) * 3 + ((int64_t)b * 3 + d) * Tt) * 2;
                int32_t m = mn[((int64_t)t * p->B + b) * 3 + d];
                for (int64_t j = 0; j < 2 * Tt; ++j) q[j] = wrap_sub(q[j], m);
            }
    }
    free(box);
    free(off);
}

/* ------------------------------------------------------------------------
 * Conditioning-token filter ("Shared negative (reference) positions").
 * A tile keeps a conditioning token when its [start,end) interval overlaps
 * the tile in all three dimensions, or when its time coordinate is negative;
 * kept tokens follow the generated ones and are shifted by the same offset.
 *
 * Readings taken: the tile's extent in dimension d is [mn, mx) of its
 * generated tokens; two half-open intervals overlap when their intersection
 * [max(s,mn), min(e,mx)) is non-empty (for non-empty intervals this is
 * s < mx && e > mn; an empty or inverted interval overlaps nothing);
 * "negative time" is start_F < 0; the test uses global (un-normalised)
 * coordinates; keep is decided per batch item; kept tokens are listed in
 * ascending k.  idx is padded with -1 past count; Kout past count is not
 * written.  kcount[b,k] is the number of tiles that kept token k; slot[t,b,k]
 * is token k's position in (t,b)'s kept list, or -1.
 * ---------------------------------------------------------------------- */
void oracle_filter(const oracle_problem *p, const int32_t *K, int32_t N,
                   const int32_t *mn, const int32_t *mx, int32_t normalize,
                   uint8_t *keep, int32_t *idx, int32_t *count, int32_t *kcount, int32_t *Kout,
                   int32_t *slot)
{
    int nt = oracle_num_tiles(p);
    for (int64_t i = 0; i < (int64_t)p->B * N; ++i) kcount[i] = 0;
    for (int t = 0; t < nt; ++t)
        for (int32_t b = 0; b < p->B; ++b) {
            int64_t tb = (int64_t)t * p->B + b;
            int32_t cnt = 0;
            for (int32_t k = 0; k < N; ++k) {
                int inside = 1;
                for (int d = 0; d < 3; ++d) {
                    int32_t s = K[(((int64_t)b * 3 + d) * N + k) * 2 + 0];
                    int32_t e = K[(((int64_t)b * 3 + d) * N + k) * 2 + 1];
                    int32_t a = s > mn[tb * 3 + d] ? s : mn[tb * 3 + d];   /* intersection   */
                    int32_t z = e < mx[tb * 3 + d] ? e : mx[tb * 3 + d];   /* [a, z) nonempty */
                    if (!(a < z)) inside = 0;
                }
                int negative_time = K[(((int64_t)b * 3 + 0) * N + k) * 2 + 0] < 0;
                int kept = inside || negative_time;
                keep[tb * N + k] = (uint8_t)kept;
                slot[tb * N + k] = kept ? cnt : -1;
                if (kept) {
                    idx[tb * N + cnt] = k;
                    for (int d = 0; d < 3; ++d)
                        for (int s = 0; s < 2; ++s) {
                            int32_t v = K[(((int64_t)b * 3 + d) * N + k) * 2 + s];
                            Kout[((tb * 3 + d) * N + cnt) * 2 + s] =
                                normalize ? wrap_sub(v, mn[tb * 3 + d]) : v;
                        }
                    kcount[(int64_t)b * N + k] += 1;
                    cnt += 1;
                }
            }
            count[tb] = cnt;
            for (int32_t k = cnt; k < N; ++k) idx[tb * N + k] = -1;
        }
}

/* ------------------------------------------------------------------------
 * Blend ("What it is": each tile output is weighted by its trapezoidal mask
 * and all tiles are summed into the full latent; the masks sum to 1).
 * Plain definition, fp64: Z = sum over tiles t (ascending) of m_t * embed(Y_t).
 * ---------------------------------------------------------------------- */
static double load_elem(const void *Y, int32_t esize, int64_t i)
{
    if (esize == 4) return (double)((const float *)Y)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)Y)[i] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

void oracle_blend(const oracle_problem *p, const void *Yout, double *Z)
{
    int nt = oracle_num_tiles(p);
    int32_t *box = (int32_t *)malloc(sizeof(int32_t) * 6 * (size_t)nt);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)nt + 1));
    oracle_plan(p, box, off);
    const int64_t T = (int64_t)p->F * p->H * p->W;
    for (int64_t i = 0; i < (int64_t)p->B * T * p->C; ++i) Z[i] = 0.0;
    for (int t = 0; t < nt; ++t) {
        const int32_t *bx = box + t * 6;
        int64_t Tt = off[t + 1] - off[t];
        for (int32_t b = 0; b < p->B; ++b) {
            int64_t j = 0;
            for (int32_t f = bx[0]; f < bx[1]; ++f)
                for (int32_t h = bx[2]; h < bx[3]; ++h)
                    for (int32_t w = bx[4]; w < bx[5]; ++w, ++j) {
                        double m = oracle_mask(p, t, f, h, w);
                        int64_t g = ((int64_t)f * p->H + h) * p->W + w;
                        int64_t src = ((int64_t)p->B * off[t] + (int64_t)b * Tt + j) * p->C;
                        for (int32_t c = 0; c < p->C; ++c)
                            Z[((int64_t)b * T + g) * p->C + c] += m * load_elem(Yout, p->esize, src + c);
                    }
        }
    }
    free(box);
    free(off);
}

/* One output cell of the blend, for sampled checks of large problems:
 * z[c] = sum over the tiles whose box holds (f,h,w) of m_t * Y_t(cell). */
void oracle_blend_cell(const oracle_problem *p, const void *Yout, int32_t b,
                       int32_t f, int32_t h, int32_t w, double *z)
{
    int nt = oracle_num_tiles(p);
    int32_t *box = (int32_t *)malloc(sizeof(int32_t) * 6 * (size_t)nt);
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * ((size_t)nt + 1));
    oracle_plan(p, box, off);
    for (int32_t c = 0; c < p->C; ++c) z[c] = 0.0;
    for (int t = 0; t < nt; ++t) {
        const int32_t *bx = box + t * 6;
        if (f < bx[0] || f >= bx[1] || h < bx[2] || h >= bx[3] || w < bx[4] || w >= bx[5]) continue;
        int64_t Tt = off[t + 1] - off[t];
        int64_t j = ((int64_t)(f - bx[0]) * (bx[3] - bx[2]) + (h - bx[2])) * (bx[5] - bx[4]) + (w - bx[4]);
        double m = oracle_mask(p, t, f, h, w);
        int64_t src = ((int64_t)p->B * off[t] + (int64_t)b * Tt + j) * p->C;
        for (int32_t c = 0; c < p->C; ++c) z[c] += m * load_elem(Yout, p->esize, src + c);
    }
    free(box);
    free(off);
}

/* ------------------------------------------------------------------------
 * Conditioning-token output reduction ("Shared negative (reference)
 * positions": a token kept by several tiles has blend weight
 * 1 / (number of tiles that kept it)).  Ycond holds each tile's outputs for its
 * kept conditioning tokens, [nt][B][ncap][C], row p of (t,b) = the p-th kept
 * token.  out[b,k,:] = sum over the tiles t that kept k (ascending) of
 * Ycond[t,b,slot,:] / n, in fp64, with n = the number of tiles that kept k
 * (kcount[b,k], the page's denominator).
 * Readings taken: a token no tile kept has no tile output; its result is 0.
 * Only ncap rows per (t,b) are stored: a tile that kept k at a position p >= ncap
 * has no stored output for it, so its term is missing from the sum, while the
 * weight of every stored term stays 1/n.
 * ---------------------------------------------------------------------- */
void oracle_cond_blend(const oracle_problem *p, int32_t N, int32_t ncap, const void *Ycond,
                       const uint8_t *keep, const int32_t *idx, const int32_t *count, double *out)
{
    int nt = oracle_num_tiles(p);
    for (int32_t b = 0; b < p->B; ++b)
        for (int32_t k = 0; k < N; ++k) {
            double *o = out + ((int64_t)b * N + k) * p->C;
            for (int32_t c = 0; c < p->C; ++c) o[c] = 0.0;
            int32_t n_keep = 0;                      /* tiles that kept k */
            for (int t = 0; t < nt; ++t) {
                int64_t tb = (int64_t)t * p->B + b;
                if (!keep[tb * N + k]) continue;
                n_keep += 1;
                int32_t pos = -1;                    /* find k in the tile's kept list */
                for (int32_t q = 0; q < count[tb]; ++q)
                    if (idx[tb * N + q] == k) { pos = q; break; }
                if (pos < 0 || pos >= ncap) continue;    /* no stored output row */
                for (int32_t c = 0; c < p->C; ++c)
                    o[c] += load_elem(Ycond, p->esize, (tb * ncap + pos) * p->C + c);
            }
            if (n_keep > 0)
                for (int32_t c = 0; c < p->C; ++c) o[c] /= (double)n_keep;
        }
}

/* ------------------------------------------------------------------------
 * Audio mean ("What it is": audio is processed untiled on every tile's forward
 * pass and averaged across tiles).  A is [nt][B][L] (L elements of one audio
 * latent per batch item); out[b,l] = (1/nt) * sum over t of A[t,b,l], fp64.
 * ---------------------------------------------------------------------- */
void oracle_tile_mean(const oracle_problem *p, const void *A, int64_t L, double *out)
{
    int nt = oracle_num_tiles(p);
    for (int64_t i = 0; i < (int64_t)p->B * L; ++i) {
        double acc = 0.0;
        for (int t = 0; t < nt; ++t) acc += load_elem(A, p->esize, (int64_t)t * p->B * L + i);
        out[i] = acc / (double)nt;
    }
}
