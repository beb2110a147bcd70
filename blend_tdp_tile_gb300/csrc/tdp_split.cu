// tdp_split.cu -- TDP tile split with tile positions and position
// normalisation ("Tiled Data Parallelism (TDP)", sections "What it is" and
// "Position normalization").
//
// Three launches on the caller's stream:
//   1. tdp_bounds_init_kernel  mn = INT32_MAX, mx = INT32_MIN        (only with positions)
//   2. tdp_bounds_kernel       per (batch, frame, 8 rows; one warp per row): min start /
//                              max end of every tile's generated tokens in those rows,
//                              positions read once, folded into mn/mx with atomics
//   3. tdp_split_kernel        scatter form: each latent row (b, f, h) is read ONCE with
//                              16-byte loads and written to every tile row that holds it
//                              (at most 2 x 2 x 2 tiles), positions likewise, shifted by
//                              mn when normalising.
// The scatter form reads the latent once instead of once per covering tile,
// so the split moves B*T*C + B*sum(T_t)*C elements, its algorithmic minimum.
#include <climits>

#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kSplitThreads = 256;
constexpr int kBoundsThreads = 256;

__global__ void tdp_bounds_init_kernel(int32_t *__restrict__ mn, int32_t *__restrict__ mx, int32_t n)
{
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        mn[i] = INT_MAX;
        mx[i] = INT_MIN;
    }
}

// Block (b, f, chunk of kBoundsRows latent rows), one warp per row.  A warp
// reads its row's positions once, 32 cells at a time (coalesced 256-byte
// loads), and reduces each W-tile segment of the 32 cells with warp min / max
// reductions (the tile loop is warp-uniform); lane 0 keeps the row's per-W-tile
// minima / maxima in the warp's own shared-memory slots (no atomics).  The
// block then combines its rows per (H-tile, W-tile, dim) and folds each result
// into the (at most 2) F-tiles holding frame f with one atomicMin / atomicMax.
constexpr int kBoundsRows = kBoundsThreads / 32;

__global__ void __launch_bounds__(kBoundsThreads)
tdp_bounds_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ P,
                  int32_t *__restrict__ mn, int32_t *__restrict__ mx)
{
    __shared__ int32_t s_mn[kBoundsRows][TDP_MAX_TILES_PER_DIM][3];
    __shared__ int32_t s_mx[kBoundsRows][TDP_MAX_TILES_PER_DIM][3];
    const int32_t nchunk = (g.H + kBoundsRows - 1) / kBoundsRows;
    const int32_t chunk = blockIdx.x % nchunk;
    const int32_t f = (blockIdx.x / nchunk) % g.F;
    const int32_t b = blockIdx.x / (nchunk * g.F);
    const int32_t h0 = chunk * kBoundsRows, h1 = min(g.H, h0 + kBoundsRows);
    const int32_t nW = g.d[2].n, nH = g.d[1].n;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t h = h0 + warp;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    const tdp_dim_geom &dW = g.d[2];

    if (h < h1) {
        for (int32_t i = lane; i < nW * 3; i += 32) {
            (&s_mn[warp][0][0])[i] = INT_MAX;
            (&s_mx[warp][0][0])[i] = INT_MIN;
        }
        __syncwarp();
        const int2 *src = P + (int64_t)b * 3 * T + ((int64_t)f * g.H + h) * g.W;
        int32_t iW = 0;
        for (int32_t wb = 0; wb < g.W; wb += 32) {
            const int32_t w = wb + lane;
            int2 v[3];
#pragma unroll
            for (int d = 0; d < 3; ++d) v[d] = w < g.W ? __ldg(src + (int64_t)d * T + w) : make_int2(INT_MAX, INT_MIN);
            while (dW.hi[iW] <= wb) ++iW;                     // first W-tile touching [wb, wb + 32)
            for (int32_t q = iW; q < nW && dW.lo[q] < wb + 32; ++q) {
                const bool in = w >= dW.lo[q] && w < dW.hi[q] && w < g.W;
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    const int32_t a = __reduce_min_sync(0xffffffffu, in ? v[d].x : INT_MAX);
                    const int32_t z = __reduce_max_sync(0xffffffffu, in ? v[d].y : INT_MIN);
                    if (lane == 0) {
                        s_mn[warp][q][d] = min(s_mn[warp][q][d], a);
                        s_mx[warp][q][d] = max(s_mx[warp][q][d], z);
                    }
                }
            }
        }
    }
    __syncthreads();
    // combine the block's rows per (H-tile, W-tile, dim) and flush
    const int32_t iHa = tdp_cover_1d(g.d[1], h0).i0;
    const tdp_cover cHz = tdp_cover_1d(g.d[1], h1 - 1);
    const int32_t iHb = cHz.i1 >= 0 ? cHz.i1 : cHz.i0;
    const tdp_cover cF = tdp_cover_1d(g.d[0], f);
    const int32_t nent = (iHb - iHa + 1) * nW * 3;
    for (int32_t i = threadIdx.x; i < nent; i += blockDim.x) {
        const int32_t iH = iHa + i / (nW * 3), iWq = (i / 3) % nW, d = i % 3;
        const int32_t rlo = max(h0, g.d[1].lo[iH]), rhi = min(h1, g.d[1].hi[iH]);
        int32_t a = INT_MAX, z = INT_MIN;
        for (int32_t r = rlo; r < rhi; ++r) {
            a = min(a, s_mn[r - h0][iWq][d]);
            z = max(z, s_mx[r - h0][iWq][d]);
        }
        if (rlo >= rhi || (a == INT_MAX && z == INT_MIN)) continue;   // nothing here (a no-op either way)
        for (int q = 0; q < 2; ++q) {
            const int32_t iF = q ? cF.i1 : cF.i0;
            if (iF < 0) break;
            const int64_t r = ((int64_t)((iF * nH + iH) * nW + iWq) * g.B + b) * 3 + d;
            atomicMin(mn + r, a);
            atomicMax(mx + r, z);
        }
    }
}

// Block = one latent row (b, f, h).  CV = 16-byte vectors per token.
__global__ void __launch_bounds__(kSplitThreads)
tdp_split_kernel(const __grid_constant__ tdp_geom g, const uint4 *__restrict__ X,
                 const int2 *__restrict__ P, int32_t normalize, uint4 *__restrict__ Y,
                 int2 *__restrict__ Q, const int32_t *__restrict__ mn)
{
    __shared__ int64_t s_tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    __shared__ int64_t s_qpos[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    __shared__ int64_t s_Tt[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    __shared__ int32_t s_tb[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];

    __shared__ int32_t s_loW[TDP_MAX_TILES_PER_DIM], s_hiW[TDP_MAX_TILES_PER_DIM];

    const int32_t row = blockIdx.x;
    const int32_t h = row % g.H, f = (row / g.H) % g.F, b = row / (g.H * g.F);
    for (int32_t i = threadIdx.x; i < g.d[2].n; i += blockDim.x) {
        s_loW[i] = g.d[2].lo[i];
        s_hiW[i] = g.d[2].hi[i];
    }
    const tdp_row_combos rc = tdp_make_combos(g, f, h);
    tdp_fill_row_table(g, rc, b, f, h, s_tok, P ? s_qpos : nullptr, P ? s_Tt : nullptr,
                       P ? s_tb : nullptr);   // ends with a barrier
    const int32_t oW = g.d[2].o;

    const int32_t nW = g.d[2].n;
    const int32_t CV = (g.C * g.esize) >> 4;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    const int64_t gtok = (int64_t)b * T + ((int64_t)f * g.H + h) * g.W;   // token of (b,f,h,0)

    // latent: every 16-byte vector of the row is loaded once and stored to each tile
    const int32_t nvec = g.W * CV;
    const uint4 *src = X + gtok * CV;
    for (int32_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int32_t w = v / CV, cv = v - w * CV;
        const uint4 x = __ldcs(src + v);
        const tdp_cover cW = tdp_cover_tab(s_loW, s_hiW, nW, g.W, oW, w);
        for (int32_t c = 0; c < rc.nc; ++c) {
            __stcs(Y + (s_tok[c * nW + cW.i0] + w) * CV + cv, x);
            if (cW.i1 >= 0) __stcs(Y + (s_tok[c * nW + cW.i1] + w) * CV + cv, x);
        }
    }
    if (!P) return;

    // positions: [B,3,T,2] -> tile-major [B,3,T_t,2], minus mn when normalising
    for (int32_t q = threadIdx.x; q < 3 * g.W; q += blockDim.x) {
        const int32_t d = q / g.W, w = q - d * g.W;
        const int2 p = __ldcs(P + ((int64_t)b * 3 + d) * T + ((int64_t)f * g.H + h) * g.W + w);
        const tdp_cover cW = tdp_cover_tab(s_loW, s_hiW, nW, g.W, oW, w);
        for (int32_t c = 0; c < rc.nc; ++c) {
            for (int32_t k = 0; k < 2; ++k) {
                const int32_t iW = k ? cW.i1 : cW.i0;
                if (iW < 0) break;
                const int32_t e = c * nW + iW;
                int2 o = p;
                if (normalize) {
                    const int32_t m = __ldg(mn + (int64_t)s_tb[e] * 3 + d);
                    o.x = (int32_t)((uint32_t)p.x - (uint32_t)m);
                    o.y = (int32_t)((uint32_t)p.y - (uint32_t)m);
                }
                __stcs(Q + s_qpos[e] + (int64_t)d * s_Tt[e] + w, o);
            }
        }
    }
}

}  // namespace

extern "C" tdp_status tdp_split(tdp_plan_t plan, const void *X, const int32_t *P, int32_t normalize,
                                void *Y, int32_t *Q, int32_t *mn, int32_t *mx, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    const bool pos = P || Q || mn || mx;
    if (pos && !(P && Q && mn && mx))
        return tdp_fail(TDP_ERR_INVALID_ARG, "P, Q, mn and mx must be all set or all NULL");
    if (g.B == 0) return tdp_ok();
    if (!X || !Y) return tdp_fail(TDP_ERR_INVALID_ARG, "null X or Y");
    if (!tdp_aligned(X, 16) || !tdp_aligned(Y, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "X and Y must be 16-byte aligned");
    if (pos && (!tdp_aligned(P, 8) || !tdp_aligned(Q, 8) || !tdp_aligned(mn, 4) || !tdp_aligned(mx, 4)))
        return tdp_fail(TDP_ERR_MISALIGNED, "P, Q need 8-byte and mn, mx 4-byte alignment");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (pos) {
        const int32_t n = g.nt * g.B * 3;
        tdp_bounds_init_kernel<<<(n + 255) / 256, 256, 0, s>>>(mn, mx, n);
        const int64_t blocks = (int64_t)g.B * g.F * ((g.H + kBoundsRows - 1) / kBoundsRows);
        tdp_bounds_kernel<<<(unsigned)blocks, kBoundsThreads, 0, s>>>(g, reinterpret_cast<const int2 *>(P), mn,
                                                                       mx);
    }
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    tdp_split_kernel<<<(unsigned)rows, kSplitThreads, 0, s>>>(
        g, reinterpret_cast<const uint4 *>(X), reinterpret_cast<const int2 *>(P), normalize,
        reinterpret_cast<uint4 *>(Y), reinterpret_cast<int2 *>(Q), mn);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
