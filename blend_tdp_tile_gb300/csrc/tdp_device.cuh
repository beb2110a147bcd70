// tdp_device.cuh -- device helpers shared by the TDP kernels: which tiles
// cover a grid coordinate, their trapezoid-ramp weights, and the per-row
// table of tile rows a latent row (b, f, h) maps to.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tdp_geom.h"

// At most two tiles cover a coordinate along one dimension (neighbours
// overlap by o and every core is at least o long).
struct tdp_cover {
    int32_t i0, i1;        // covering tiles, i0 < i1; i1 = -1 when only one
    int32_t num0, num1;    // ramp numerators over den = o + 1
};

// Tiles covering coordinate x in [0, L) and their ramp numerators
// ("Tiled Data Parallelism (TDP)", "What it is": trapezoidal masks summing to
// one).  Across the o-cell overlap of tiles i, i+1, with k = x - lo[i+1], the
// right tile weighs (k+1)/(o+1) and the left one (o-k)/(o+1).  lo/hi may live in
// shared memory (lanes with different x then read them in parallel) or in the
// kernel parameters.  32-bit arithmetic: the plan keeps L * (n + 1) below 2^32.
__device__ __forceinline__ tdp_cover tdp_cover_tab(const int32_t *lo, const int32_t *hi, int32_t n, int32_t L,
                                                   int32_t o, int32_t x)
{
    // core index: the largest i with floor(i*L/n) <= x, i.e. ceil((x+1)*n/L) - 1
    const int32_t ci = (int32_t)(((uint32_t)(x + 1) * (uint32_t)n + (uint32_t)(L - 1)) / (uint32_t)L) - 1;
    tdp_cover c;
    if (ci > 0 && x < hi[ci - 1]) {
        const int32_t k = x - lo[ci];
        c.i0 = ci - 1;
        c.i1 = ci;
        c.num0 = o - k;
        c.num1 = k + 1;
    } else if (ci < n - 1 && x >= lo[ci + 1]) {
        const int32_t k = x - lo[ci + 1];
        c.i0 = ci;
        c.i1 = ci + 1;
        c.num0 = o - k;
        c.num1 = k + 1;
    } else {
        c.i0 = ci;
        c.i1 = -1;
        c.num0 = o + 1;
        c.num1 = 0;
    }
    return c;
}

__device__ __forceinline__ tdp_cover tdp_cover_1d(const tdp_dim_geom &dg, int32_t x)
{
    return tdp_cover_tab(dg.lo, dg.hi, dg.n, dg.L, dg.o, x);
}

// fp32 ramp weight num/(o+1), IEEE round-to-nearest division.
__device__ __forceinline__ float tdp_weight(int32_t num, int32_t o)
{
    return __fdiv_rn((float)num, (float)(o + 1));
}

// ---------------------------------------------------------------------------
// Row table.  A latent row (b, f, h) lies in at most 2 F-tiles x 2 H-tiles
// ("combos", in ascending (iF, iH)); inside each combo every W-tile iW holds a
// contiguous run of that row.  For combo c and W-tile iW:
//   tok[c][iW]  token index, in the tile-major buffers, of the row's cell w = 0
//               (so cell w sits at tok + w; only w in [lo_W, hi_W) is used)
//   qpos[c][iW] same for the tile-major position buffer, d = 0 (add d*T_t)
//   Tt[c][iW]   tokens of the tile
//   tb[c][iW]   t*B + b (row of mn/mx)
// ---------------------------------------------------------------------------
#define TDP_MAX_COMBOS 4

struct tdp_row_combos {
    int32_t nc;                           // combos (1, 2 or 4)
    int32_t nH;                           // H-tiles per F-tile in the row (1 or 2)
    int32_t iF0, iF1, iH0, iH1;           // covering F- and H-tiles (second = -1 when none)
    float rF0, rF1, rH0, rH1;             // their ramp weights
    // Combo c in ascending (iF, iH): F-tile c / nH, H-tile c % nH.  Scalars and selects
    // rather than arrays, so that a combo index known only at run time needs no local memory.
    __device__ __forceinline__ int32_t fsel(int32_t c) const { return nH == 2 ? c >> 1 : c; }
    __device__ __forceinline__ int32_t hsel(int32_t c) const { return nH == 2 ? c & 1 : 0; }
    __device__ __forceinline__ int32_t iF(int32_t c) const { return fsel(c) ? iF1 : iF0; }
    __device__ __forceinline__ int32_t iH(int32_t c) const { return hsel(c) ? iH1 : iH0; }
    // r_F * r_H of combo c
    __device__ __forceinline__ float rFH(int32_t c) const { return (fsel(c) ? rF1 : rF0) * (hsel(c) ? rH1 : rH0); }
};

__device__ __forceinline__ tdp_row_combos tdp_make_combos(const tdp_geom &g, int32_t f, int32_t h)
{
    const tdp_cover cF = tdp_cover_1d(g.d[0], f);
    const tdp_cover cH = tdp_cover_1d(g.d[1], h);
    tdp_row_combos rc;
    const int32_t nF = cF.i1 >= 0 ? 2 : 1;
    rc.nH = cH.i1 >= 0 ? 2 : 1;
    rc.nc = nF * rc.nH;
    rc.iF0 = cF.i0;
    rc.iF1 = cF.i1;
    rc.iH0 = cH.i0;
    rc.iH1 = cH.i1;
    rc.rF0 = tdp_weight(cF.num0, g.d[0].o);
    rc.rF1 = tdp_weight(cF.num1, g.d[0].o);
    rc.rH0 = tdp_weight(cH.num0, g.d[1].o);
    rc.rH1 = tdp_weight(cH.num1, g.d[1].o);
    return rc;
}

// Token offset off_t of tile (iF, iH, iW) in the tile-major buffers.
__device__ __forceinline__ int64_t tdp_tile_off(const tdp_geom &g, int32_t iF, int32_t iH, int32_t iW)
{
    const int64_t SF = g.d[0].hi[iF] - g.d[0].lo[iF];
    const int64_t SH = g.d[1].hi[iH] - g.d[1].lo[iH];
    return (int64_t)g.d[0].pre[iF] * g.d[1].sum * g.d[2].sum +
           SF * ((int64_t)g.d[1].pre[iH] * g.d[2].sum + SH * (int64_t)g.d[2].pre[iW]);
}

// Fill tok / qpos / Tt / tb (each [TDP_MAX_COMBOS * nW]) for row (b, f, h); entry c*nW + iW.
// Called by the whole block; ends with __syncthreads().
__device__ __forceinline__ void tdp_fill_row_table(const tdp_geom &g, const tdp_row_combos &rc,
                                                   int32_t b, int32_t f, int32_t h,
                                                   int64_t *tok, int64_t *qpos, int64_t *Tt,
                                                   int32_t *tb)
{
    const int32_t nW = g.d[2].n;
    for (int32_t e = threadIdx.x; e < rc.nc * nW; e += blockDim.x) {
        const int32_t c = e / nW, iW = e % nW;
        const int32_t iF = rc.iF(c), iH = rc.iH(c);
        const int64_t SH = g.d[1].hi[iH] - g.d[1].lo[iH];
        const int64_t SW = g.d[2].hi[iW] - g.d[2].lo[iW];
        const int64_t SF = g.d[0].hi[iF] - g.d[0].lo[iF];
        const int64_t T = SF * SH * SW;
        const int64_t off = tdp_tile_off(g, iF, iH, iW);
        const int64_t jrow = ((int64_t)(f - g.d[0].lo[iF]) * SH + (h - g.d[1].lo[iH])) * SW - g.d[2].lo[iW];
        tok[e] = (int64_t)g.B * off + (int64_t)b * T + jrow;
        if (qpos) qpos[e] = (int64_t)g.B * off * 3 + (int64_t)b * 3 * T + jrow;
        if (Tt) Tt[e] = T;
        if (tb) tb[e] = ((iF * g.d[1].n + iH) * nW + iW) * g.B + b;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32 on 16-byte vectors (8 bf16 or 4 fp32 per uint4).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float tdp_bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float tdp_bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two fp32 -> packed bf16x2 (round to nearest even), low half = `lo`.
__device__ __forceinline__ uint32_t tdp_pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The kernels of the library let the next
// kernel in their stream launch early (tdp_pdl_trigger at their start; the two
// latency-bound filter kernels instead let it launch as their blocks exit), and
// every kernel waits for the kernel before it to complete, with its memory
// visible, before it touches global memory that kernel may write (tdp_pdl_wait).  The work before
// the wait is limited to kernel parameters and shared memory, except where a
// kernel is launched only behind a kernel of this library whose own wait comes
// first (stated at each such kernel).  Both are no-ops for a plain launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tdp_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void tdp_pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
