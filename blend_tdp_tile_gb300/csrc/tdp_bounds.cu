// tdp_bounds.cu -- the position extent of every tile: minimum start and
// maximum end of its generated tokens, per batch item and dimension
// ("Tiled Data Parallelism (TDP)", section "Position normalization": the
// offset is gen_pos[..., 0].amin over the tile's tokens; the maximum end is the
// tile's far edge for the conditioning filter).
//
// Two launches on the caller's stream:
//   1. tdp_bounds_init_kernel  mn = INT32_MAX, mx = INT32_MIN (a plain launch: it starts
//                              once all earlier work in the stream has completed)
//   2. tdp_bounds_kernel       per (batch, frame, 8 rows; one warp per row): min start /
//                              max end of every tile's generated tokens in those rows,
//                              positions read once, folded into mn/mx with atomics.
//                              A programmatic dependent launch behind the init kernel:
//                              the row reductions, which read only the positions, run
//                              while the init kernel finishes; the atomics wait for it.
#include <climits>

#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kBoundsThreads = 256;

__global__ void tdp_bounds_init_kernel(int32_t *__restrict__ mn, int32_t *__restrict__ mx, int32_t n)
{
    tdp_pdl_trigger();
    tdp_pdl_wait();
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
constexpr int kBoundsChunks = 4;     // 32-cell chunks of a row whose loads a warp keeps in flight

__global__ void __launch_bounds__(kBoundsThreads)
tdp_bounds_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ P,
                  int32_t *__restrict__ mn, int32_t *__restrict__ mx)
{
    __shared__ int32_t s_mn[kBoundsRows][TDP_MAX_TILES_PER_DIM][3];
    __shared__ int32_t s_mx[kBoundsRows][TDP_MAX_TILES_PER_DIM][3];
    tdp_pdl_trigger();
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
        for (int32_t wb0 = 0; wb0 < g.W; wb0 += 32 * kBoundsChunks) {
            // loads of kBoundsChunks 32-cell chunks (3 dims each) in flight at once
            int2 v[kBoundsChunks][3];
#pragma unroll
            for (int u = 0; u < kBoundsChunks; ++u) {
                const int32_t w = wb0 + 32 * u + lane;
#pragma unroll
                for (int d = 0; d < 3; ++d)
                    v[u][d] = w < g.W ? __ldg(src + (int64_t)d * T + w) : make_int2(INT_MAX, INT_MIN);
            }
#pragma unroll
            for (int u = 0; u < kBoundsChunks; ++u) {
                const int32_t wb = wb0 + 32 * u;
                if (wb >= g.W) break;                             // warp-uniform
                const int32_t w = wb + lane;
                while (dW.hi[iW] <= wb) ++iW;                     // first W-tile touching [wb, wb + 32)
                for (int32_t q = iW; q < nW && dW.lo[q] < wb + 32; ++q) {
                    const bool in = w >= dW.lo[q] && w < dW.hi[q] && w < g.W;
#pragma unroll
                    for (int d = 0; d < 3; ++d) {
                        const int32_t a = __reduce_min_sync(0xffffffffu, in ? v[u][d].x : INT_MAX);
                        const int32_t z = __reduce_max_sync(0xffffffffu, in ? v[u][d].y : INT_MIN);
                        if (lane == 0) {
                            s_mn[warp][q][d] = min(s_mn[warp][q][d], a);
                            s_mx[warp][q][d] = max(s_mx[warp][q][d], z);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    // Positions were read before the wait: this kernel is only launched right behind
    // tdp_bounds_init_kernel, a plain launch, so every earlier writer of P has completed.
    tdp_pdl_wait();                                   // mn / mx initialised
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

}  // namespace

cudaError_t tdp_launch_bounds(const tdp_geom &g, const int32_t *P, int32_t *mn, int32_t *mx, cudaStream_t s)
{
    const int32_t n = g.nt * g.B * 3;
    cudaError_t err = tdp_launch(false, tdp_bounds_init_kernel, (unsigned)((n + 255) / 256), 256, s, mn, mx, n);
    const int64_t blocks = (int64_t)g.B * g.F * ((g.H + kBoundsRows - 1) / kBoundsRows);
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_bounds_kernel, (unsigned)blocks, kBoundsThreads, s, g,
                         reinterpret_cast<const int2 *>(P), mn, mx);
    return err;
}

extern "C" tdp_status tdp_pos_bounds(tdp_plan_t plan, const int32_t *P, int32_t *mn, int32_t *mx,
                                     tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (g.B == 0) return tdp_ok();
    if (!P || !mn || !mx) return tdp_fail(TDP_ERR_INVALID_ARG, "null P, mn or mx");
    if (!tdp_aligned(P, 8) || !tdp_aligned(mn, 4) || !tdp_aligned(mx, 4))
        return tdp_fail(TDP_ERR_MISALIGNED, "P needs 8-byte and mn, mx 4-byte alignment");
    cudaError_t err = tdp_launch_bounds(g, P, mn, mx, reinterpret_cast<cudaStream_t>(stream));
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
