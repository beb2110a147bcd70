// tdp_split.cu -- TDP tile split with tile positions and position
// normalisation ("Tiled Data Parallelism (TDP)", sections "What it is" and
// "Position normalization").
//
// One launch, tdp_split_kernel, in scatter form: each latent row (b, f, h) is
// read ONCE with 16-byte loads and written to every tile row that holds it
// (at most 2 x 2 x 2 tiles); its positions likewise, shifted by the tiles'
// mn (from tdp_pos_bounds) when normalising.
// The scatter form reads the latent once instead of once per covering tile,
// so the split moves B*T*C + B*sum(T_t)*C elements, its algorithmic minimum.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitUnroll = 4;      // latent vectors each thread loads before storing any

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
    for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += kSplitUnroll * blockDim.x) {
        uint4 xs[kSplitUnroll];                     // kSplitUnroll loads in flight per thread
#pragma unroll
        for (int u = 0; u < kSplitUnroll; ++u) {
            const int32_t v = v0 + u * blockDim.x;
            if (v < nvec) xs[u] = __ldcs(src + v);
        }
#pragma unroll
        for (int u = 0; u < kSplitUnroll; ++u) {
            const int32_t v = v0 + u * blockDim.x;
            if (v >= nvec) break;
            const int32_t w = v / CV, cv = v - w * CV;
            const tdp_cover cW = tdp_cover_tab(s_loW, s_hiW, nW, g.W, oW, w);
            for (int32_t c = 0; c < rc.nc; ++c) {
                __stcs(Y + (s_tok[c * nW + cW.i0] + w) * CV + cv, xs[u]);
                if (cW.i1 >= 0) __stcs(Y + (s_tok[c * nW + cW.i1] + w) * CV + cv, xs[u]);
            }
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
                Q[s_qpos[e] + (int64_t)d * s_Tt[e] + w] = o;   // default policy: neighbouring rows merge in L2
            }
        }
    }
}

}  // namespace

extern "C" tdp_status tdp_split(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *mn,
                                int32_t normalize, void *Y, int32_t *Q, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if ((P == nullptr) != (Q == nullptr)) return tdp_fail(TDP_ERR_INVALID_ARG, "P and Q must be both set or both NULL");
    if (P && normalize && !mn) return tdp_fail(TDP_ERR_INVALID_ARG, "normalising needs mn");
    if (g.B == 0) return tdp_ok();
    if (!X || !Y) return tdp_fail(TDP_ERR_INVALID_ARG, "null X or Y");
    if (!tdp_aligned(X, 16) || !tdp_aligned(Y, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "X and Y must be 16-byte aligned");
    if (P && (!tdp_aligned(P, 8) || !tdp_aligned(Q, 8) || !tdp_aligned(mn, 4)))
        return tdp_fail(TDP_ERR_MISALIGNED, "P, Q need 8-byte and mn 4-byte alignment");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    tdp_split_kernel<<<(unsigned)rows, kSplitThreads, 0, s>>>(
        g, reinterpret_cast<const uint4 *>(X), reinterpret_cast<const int2 *>(P), P ? normalize : 0,
        reinterpret_cast<uint4 *>(Y), reinterpret_cast<int2 *>(Q), mn);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
