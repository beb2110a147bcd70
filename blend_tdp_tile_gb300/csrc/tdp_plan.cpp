// tdp_plan.cpp -- host-side plan: validation and tile geometry of a TDP
// problem ("Tiled Data Parallelism (TDP)", "API / Tiling config").  No CUDA
// call is made here.
#include <stdlib.h>
#include <string.h>

#include <new>
#include <string>

#include "tdp.h"
#include "tdp_internal.h"

namespace {
thread_local std::string g_detail;
}

tdp_status tdp_fail(tdp_status st, const char *detail)
{
    g_detail = detail ? detail : "";
    return st;
}

tdp_status tdp_ok()
{
    g_detail.clear();
    return TDP_OK;
}

namespace {

// Fill one dimension's boxes.  Returns false for an invalid (L, n, o).
bool make_dim(int32_t L, int32_t n, int32_t o, tdp_dim_geom *dg, std::string *why)
{
    if (n < 1 || o < 0 || L < 1 || n > L) {
        *why = "need 1 <= num_tiles <= extent and overlap >= 0";
        return false;
    }
    if (n > TDP_MAX_TILES_PER_DIM) {
        *why = "num_tiles above TDP_MAX_TILES_PER_DIM";
        return false;
    }
    if (n == 1) o = 0;
    if (n >= 2 && L / n < o) {
        *why = "overlap longer than the shortest core floor(extent/num_tiles)";
        return false;
    }
    memset(dg, 0, sizeof(*dg));
    dg->L = L;
    dg->n = n;
    dg->o = o;
    const int32_t left = o / 2, right = o - left;
    int32_t acc = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t c0 = (int32_t)(((int64_t)i * L) / n);
        const int32_t c1 = (int32_t)(((int64_t)(i + 1) * L) / n);
        dg->lo[i] = i > 0 ? c0 - left : 0;
        dg->hi[i] = i < n - 1 ? c1 + right : L;
        dg->pre[i] = acc;
        acc += dg->hi[i] - dg->lo[i];
    }
    dg->sum = acc;
    // The 1-D weights (ramp numerators over o+1) must sum to o+1 at every cell.
    for (int32_t x = 0; x < L; ++x) {
        int32_t s = 0;
        for (int32_t i = 0; i < n; ++i) {
            if (x < dg->lo[i] || x >= dg->hi[i]) continue;
            if (i > 0 && x < dg->hi[i - 1]) s += x - dg->lo[i] + 1;
            else if (i < n - 1 && x >= dg->lo[i + 1]) s += o - (x - dg->lo[i + 1]);
            else s += o + 1;
        }
        if (s != o + 1) {
            *why = "masks do not sum to one";
            return false;
        }
    }
    return true;
}

}  // namespace

extern "C" tdp_status tdp_plan_create(const tdp_problem *prob, tdp_plan_t *out)
{
    if (!prob || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null argument");
    if (prob->dtype != TDP_F32 && prob->dtype != TDP_BF16)
        return tdp_fail(TDP_ERR_UNSUPPORTED_DTYPE, "dtype must be TDP_F32 or TDP_BF16");
    if (prob->B < 0 || prob->C < 1 || prob->F < 1 || prob->H < 1 || prob->W < 1)
        return tdp_fail(TDP_ERR_INVALID_ARG, "need B >= 0 and C, F, H, W >= 1");
    if (prob->F > (1 << 25) || prob->H > (1 << 25) || prob->W > (1 << 25))
        return tdp_fail(TDP_ERR_TOO_LARGE, "F, H and W must be at most 2^25");
    const int32_t esize = prob->dtype == TDP_F32 ? 4 : 2;
    if (((int64_t)prob->C * esize) % 16 != 0)
        return tdp_fail(TDP_ERR_MISALIGNED, "C * element size must be a multiple of 16 bytes");

    tdp_geom g;
    memset(&g, 0, sizeof(g));
    g.B = prob->B;
    g.F = prob->F;
    g.H = prob->H;
    g.W = prob->W;
    g.C = prob->C;
    g.dtype = prob->dtype;
    g.esize = esize;
    const int32_t L[3] = {prob->F, prob->H, prob->W};
    std::string why;
    for (int d = 0; d < 3; ++d) {
        if (!make_dim(L[d], prob->dim[d].num_tiles, prob->dim[d].overlap, &g.d[d], &why)) {
            const char *names[3] = {"F: ", "H: ", "W: "};
            std::string msg = std::string(names[d]) + why;
            return tdp_fail(why.find("TDP_MAX") != std::string::npos ? TDP_ERR_TOO_LARGE
                                                                      : TDP_ERR_BAD_GEOMETRY,
                            msg.c_str());
        }
    }
    g.nt = g.d[0].n * g.d[1].n * g.d[2].n;
    g.total = (int64_t)g.d[0].sum * g.d[1].sum * g.d[2].sum;
    // Element indices are int64 in every kernel; keep the largest buffer well inside it,
    // and the per-row token count inside int32.
    const int64_t tiles_elems = (int64_t)g.B * g.total * g.C;
    const int64_t latent_elems = (int64_t)g.B * g.F * g.H * g.W * g.C;
    if (g.total > ((int64_t)1 << 40) || tiles_elems > ((int64_t)1 << 56) ||
        latent_elems > ((int64_t)1 << 56) || (int64_t)g.B * g.F * g.H > 0x7fffffffLL ||
        (int64_t)g.W * g.C > 0x7fffffffLL || (int64_t)g.nt * g.B * 3 > 0x7fffffffLL)
        return tdp_fail(TDP_ERR_TOO_LARGE, "problem exceeds index ranges");

    // The kernels locate tile (iF, iH, iW) with the closed form
    //   off = pre_F*sum_H*sum_W + S_F*(pre_H*sum_W + S_H*pre_W);
    // check it against the running sum of tile sizes in tile order.
    {
        int64_t acc = 0;
        for (int32_t iF = 0; iF < g.d[0].n; ++iF)
            for (int32_t iH = 0; iH < g.d[1].n; ++iH)
                for (int32_t iW = 0; iW < g.d[2].n; ++iW) {
                    const int64_t SF = g.d[0].hi[iF] - g.d[0].lo[iF];
                    const int64_t SH = g.d[1].hi[iH] - g.d[1].lo[iH];
                    const int64_t SW = g.d[2].hi[iW] - g.d[2].lo[iW];
                    const int64_t off = (int64_t)g.d[0].pre[iF] * g.d[1].sum * g.d[2].sum +
                                        SF * ((int64_t)g.d[1].pre[iH] * g.d[2].sum + SH * g.d[2].pre[iW]);
                    if (off != acc) return tdp_fail(TDP_ERR_BAD_GEOMETRY, "internal: tile offsets inconsistent");
                    acc += SF * SH * SW;
                }
        if (acc != g.total) return tdp_fail(TDP_ERR_BAD_GEOMETRY, "internal: tile token total inconsistent");
    }

    tdp_plan_s *p = new (std::nothrow) tdp_plan_s;
    if (!p) return tdp_fail(TDP_ERR_INVALID_ARG, "out of host memory");
    p->g = g;
    *out = p;
    return tdp_ok();
}

extern "C" tdp_status tdp_plan_info(tdp_plan_t plan, int32_t *n_tiles, int64_t *total_tile_tokens,
                                    int32_t *boxes, int64_t *offsets)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (n_tiles) *n_tiles = g.nt;
    if (total_tile_tokens) *total_tile_tokens = g.total;
    const int32_t nH = g.d[1].n, nW = g.d[2].n;
    int64_t acc = 0;
    for (int32_t t = 0; t < g.nt; ++t) {
        const int32_t i[3] = {t / (nH * nW), (t / nW) % nH, t % nW};
        int64_t tt = 1;
        for (int d = 0; d < 3; ++d) {
            if (boxes) {
                boxes[(t * 3 + d) * 2 + 0] = g.d[d].lo[i[d]];
                boxes[(t * 3 + d) * 2 + 1] = g.d[d].hi[i[d]];
            }
            tt *= g.d[d].hi[i[d]] - g.d[d].lo[i[d]];
        }
        if (offsets) offsets[t] = acc;
        acc += tt;
    }
    if (offsets) offsets[g.nt] = acc;
    return tdp_ok();
}

extern "C" void tdp_plan_destroy(tdp_plan_t plan)
{
    delete plan;
}

extern "C" const char *tdp_status_str(tdp_status s)
{
    switch (s) {
    case TDP_OK: return "TDP_OK";
    case TDP_ERR_INVALID_ARG: return "TDP_ERR_INVALID_ARG";
    case TDP_ERR_BAD_GEOMETRY: return "TDP_ERR_BAD_GEOMETRY";
    case TDP_ERR_UNSUPPORTED_DTYPE: return "TDP_ERR_UNSUPPORTED_DTYPE";
    case TDP_ERR_MISALIGNED: return "TDP_ERR_MISALIGNED";
    case TDP_ERR_TOO_LARGE: return "TDP_ERR_TOO_LARGE";
    case TDP_ERR_CUDA: return "TDP_ERR_CUDA";
    }
    return "TDP_ERR_UNKNOWN";
}

extern "C" const char *tdp_last_error_detail(void)
{
    return g_detail.c_str();
}

extern "C" tdp_status tdp_balanced_tile_split(int32_t world, int32_t *h_tiles, int32_t *w_tiles)
{
    if (world < 1 || !h_tiles || !w_tiles) return tdp_fail(TDP_ERR_INVALID_ARG, "need world >= 1 and outputs");
    int32_t best = 1;
    for (int32_t h = 1; (int64_t)h * h <= world; ++h)
        if (world % h == 0) best = h;    // the largest divisor <= sqrt(world)
    *h_tiles = best;
    *w_tiles = world / best;
    return tdp_ok();
}

extern "C" tdp_status tdp_tiles_for_size(int32_t L, int32_t tile_size, int32_t overlap, int32_t *num_tiles)
{
    if (!num_tiles || L < 1 || tile_size < 1 || overlap < 0)
        return tdp_fail(TDP_ERR_INVALID_ARG, "need L, tile_size >= 1, overlap >= 0 and an output");
    const int32_t nmax = L < TDP_MAX_TILES_PER_DIM ? L : TDP_MAX_TILES_PER_DIM;
    std::string why;
    for (int32_t n = 1; n <= nmax; ++n) {
        tdp_dim_geom dg;
        if (!make_dim(L, n, overlap, &dg, &why)) continue;
        int32_t largest = 0;
        for (int32_t i = 0; i < n; ++i) largest = dg.hi[i] - dg.lo[i] > largest ? dg.hi[i] - dg.lo[i] : largest;
        if (largest <= tile_size) {
            *num_tiles = n;
            return tdp_ok();
        }
    }
    return tdp_fail(TDP_ERR_BAD_GEOMETRY, "no valid tile count gives tiles that small");
}

extern "C" tdp_status tdp_rank_tiles(tdp_plan_t plan, int32_t rank, int32_t world, int32_t *tiles, int32_t *n)
{
    if (!plan || !n || world < 1 || rank < 0 || rank >= world)
        return tdp_fail(TDP_ERR_INVALID_ARG, "need a plan, an output and 0 <= rank < world");
    int32_t k = 0;
    for (int32_t t = rank; t < plan->g.nt; t += world) {
        if (tiles) tiles[k] = t;
        ++k;
    }
    *n = k;
    return tdp_ok();
}
