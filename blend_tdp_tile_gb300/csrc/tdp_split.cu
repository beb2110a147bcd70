// tdp_split.cu -- TDP tile split with tile positions and position
// normalisation ("Tiled Data Parallelism (TDP)", sections "What it is" and
// "Position normalization").
//
// Three launches on the caller's stream:
//   1. tdp_bounds_init_kernel  mn = INT32_MAX, mx = INT32_MIN        (only with positions)
//   2. tdp_bounds_kernel       per (tile, batch, tile-frame): min start / max end of the
//                              tile's generated tokens, folded into mn/mx with atomics
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

// Block (t, b, fl): the tile-local frame fl of tile t, batch item b.  Reduces all
// three dimensions over the frame's SH x SW tokens (every thread keeps
// 3 * kBoundsUnroll loads in flight), then 6 atomics.
constexpr int kBoundsUnroll = 4;

__global__ void __launch_bounds__(kBoundsThreads)
tdp_bounds_kernel(const __grid_constant__ tdp_geom g, int32_t max_sf, const int2 *__restrict__ P,
                  int32_t *__restrict__ mn, int32_t *__restrict__ mx)
{
    const int32_t fl = blockIdx.x % max_sf;
    const int32_t tb = blockIdx.x / max_sf;          // t*B + b
    const int32_t t = tb / g.B, b = tb % g.B;
    const int32_t nH = g.d[1].n, nW = g.d[2].n;
    const int32_t iF = t / (nH * nW), iH = (t / nW) % nH, iW = t % nW;
    const int32_t loF = g.d[0].lo[iF], SF = g.d[0].hi[iF] - loF;
    if (fl >= SF) return;
    const int32_t loH = g.d[1].lo[iH], SH = g.d[1].hi[iH] - loH;
    const int32_t loW = g.d[2].lo[iW], SW = g.d[2].hi[iW] - loW;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    const int32_t f = loF + fl;
    const int2 *src0 = P + (int64_t)b * 3 * T + ((int64_t)f * g.H + loH) * g.W + loW;

    int32_t lo[3] = {INT_MAX, INT_MAX, INT_MAX}, hi[3] = {INT_MIN, INT_MIN, INT_MIN};
    const int32_t n = SH * SW;
    for (int32_t e0 = threadIdx.x; e0 < n; e0 += kBoundsUnroll * blockDim.x) {
        int2 v[kBoundsUnroll][3];
#pragma unroll
        for (int u = 0; u < kBoundsUnroll; ++u) {
            const int32_t e = e0 + u * blockDim.x;
            if (e < n) {
                const int32_t hh = e / SW, ww = e - hh * SW;
                const int64_t off = (int64_t)hh * g.W + ww;
#pragma unroll
                for (int d = 0; d < 3; ++d) v[u][d] = __ldg(src0 + d * T + off);
            } else {
#pragma unroll
                for (int d = 0; d < 3; ++d) v[u][d] = make_int2(INT_MAX, INT_MIN);
            }
        }
#pragma unroll
        for (int u = 0; u < kBoundsUnroll; ++u)
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                lo[d] = min(lo[d], v[u][d].x);
                hi[d] = max(hi[d], v[u][d].y);
            }
    }
    __shared__ int32_t s_mn[3][kBoundsThreads / 32], s_mx[3][kBoundsThreads / 32];
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const int32_t a = __reduce_min_sync(0xffffffffu, lo[d]);
        const int32_t z = __reduce_max_sync(0xffffffffu, hi[d]);
        if (lane == 0) {
            s_mn[d][warp] = a;
            s_mx[d][warp] = z;
        }
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        const int32_t d = threadIdx.x;
        int32_t a = INT_MAX, z = INT_MIN;
        for (int32_t w = 0; w < kBoundsThreads / 32; ++w) {
            a = min(a, s_mn[d][w]);
            z = max(z, s_mx[d][w]);
        }
        atomicMin(mn + (int64_t)tb * 3 + d, a);
        atomicMax(mx + (int64_t)tb * 3 + d, z);
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

    const int32_t row = blockIdx.x;
    const int32_t h = row % g.H, f = (row / g.H) % g.F, b = row / (g.H * g.F);
    const tdp_row_combos rc = tdp_make_combos(g, f, h);
    tdp_fill_row_table(g, rc, b, f, h, s_tok, P ? s_qpos : nullptr, P ? s_Tt : nullptr,
                       P ? s_tb : nullptr);

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
        const tdp_cover cW = tdp_cover_1d(g.d[2], w);
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
        const tdp_cover cW = tdp_cover_1d(g.d[2], w);
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
        int32_t max_sf = 0;
        for (int32_t i = 0; i < g.d[0].n; ++i) max_sf = max(max_sf, g.d[0].hi[i] - g.d[0].lo[i]);
        const int64_t blocks = (int64_t)g.nt * g.B * max_sf;
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "bounds grid too large");
        tdp_bounds_kernel<<<(unsigned)blocks, kBoundsThreads, 0, s>>>(
            g, max_sf, reinterpret_cast<const int2 *>(P), mn, mx);
    }
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    tdp_split_kernel<<<(unsigned)rows, kSplitThreads, 0, s>>>(
        g, reinterpret_cast<const uint4 *>(X), reinterpret_cast<const int2 *>(P), normalize,
        reinterpret_cast<uint4 *>(Y), reinterpret_cast<int2 *>(Q), mn);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
