// tdp_cond.cu -- the two reductions over tiles besides the latent blend
// ("Tiled Data Parallelism (TDP)"):
//   tdp_cond_blend_rows_kernel, tdp_cond_blend_kernel
//                          each conditioning token's per-tile outputs averaged
//                          over the tiles that kept it ("Shared negative
//                          (reference) positions": weight 1/(tiles that kept it));
//   tdp_tile_mean_kernel   the audio latent averaged over all tiles ("What it
//                          is": audio is processed on every tile and averaged).
// Both are gather form and accumulate in fp32; no atomics, no scratch.  The
// conditioning blend adds each token's rows in ascending tile order, one after
// another; the tile mean adds the tiles of each quarter of the tile range in
// ascending order and then the four quarters' sums in order.
//
// tdp_cond_blend has two kernels.  With at most kStageTiles tiles (and rows of
// Ycond numbered below 2^32), tdp_cond_blend_rows_kernel runs the block routine of
// tdp_cond_rows.cuh, kTok tokens per block.  With more tiles, tdp_cond_blend_kernel
// gives each token a warp, which reads the token's slots 32 tiles at a time.
#include "tdp.h"
#include "tdp_cond_rows.cuh"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

using namespace tdp_cr;

constexpr int kThreads = 256;
constexpr int kMeanVecs = 64;     // output vectors per tile-mean block
constexpr int kMeanParts = 4;     // threads per output vector, each over a quarter of the tiles
constexpr int kMeanUnroll = 8;    // tile loads a tile-mean thread keeps in flight

// Warp = one conditioning token (b, k).  Per round of 32 tiles, lane l loads the
// token's slot in tile t0 + l; a ballot gives the tiles that kept it, in
// ascending order, and their rows (lanes across the channel vectors) are loaded
// up to kRowsInFlight at a time and added to the sum in that order.
constexpr int kRowsInFlight = 4;

template <int BF16>
__global__ void __launch_bounds__(kThreads)
tdp_cond_blend_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV,
                      const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot, uint4 *__restrict__ out)
{
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (tok >= (int64_t)g.B * N) return;                 // warp-uniform
    const int32_t b = (int32_t)(tok / N), k = (int32_t)(tok - (int64_t)b * N);
    for (int32_t cv0 = 0; cv0 < CV; cv0 += 32) {
        const int32_t cv = cv0 + lane;
        const bool act = cv < CV;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int32_t den = 0;                                     // tiles that kept the token
        for (int32_t t0 = 0; t0 < g.nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < g.nt ? __ldg(slot + ((int64_t)t * g.B + b) * N + k) : -1;
            den += __popc(__ballot_sync(0xffffffffu, sl >= 0));
            uint32_t m = __ballot_sync(0xffffffffu, sl >= 0 && sl < ncap);
            while (m) {                                      // warp-uniform
                uint4 y[kRowsInFlight];
                int32_t got = 0;
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u) {
                    if (m) {
                        const int32_t j = __ffs(m) - 1;
                        m &= m - 1;
                        const int32_t sj = __shfl_sync(0xffffffffu, sl, j);
                        const int64_t tb = (int64_t)(t0 + j) * g.B + b;
                        if (act) y[u] = __ldcs(Ycond + (tb * ncap + sj) * CV + cv);
                        got = u + 1;
                    }
                }
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u)
                    if (u < got && act) acc_add<BF16>(acc, y[u]);
            }
        }
        if (act) __stcs(out + tok * CV + cv, den > 0 ? acc_weigh<BF16>(acc, (float)den) : make_uint4(0u, 0u, 0u, 0u));
    }
}

// Block = tokens k0 .. k0 + kTok - 1 of batch item b.
template <int BF16>
__global__ void __launch_bounds__(kTokThreads, kTokMinBlocks)
tdp_cond_blend_rows_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV,
                           const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot,
                           uint4 *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    cond_rows_block<BF16>(g, N, ncap, CV, Ycond, slot, out, blockIdx.x, dsm);
}

// Block = kMeanVecs output vectors of out[B, L]; thread (part p, vector v) sums
// tiles [p*nt/4, (p+1)*nt/4) in ascending order, kMeanUnroll loads in flight;
// part 0 adds the four sums in order and multiplies by the weight 1/nt.
template <int BF16>
__global__ void __launch_bounds__(kMeanVecs * kMeanParts)
tdp_tile_mean_kernel(int32_t nt, int64_t nvec, const uint4 *__restrict__ A, uint4 *__restrict__ out)
{
    __shared__ float s_part[kMeanParts][8][kMeanVecs];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t vi = threadIdx.x % kMeanVecs, p = threadIdx.x / kMeanVecs;
    const int64_t v = (int64_t)blockIdx.x * kMeanVecs + vi;
    const int32_t ta = (int32_t)((int64_t)p * nt / kMeanParts), tz = (int32_t)((int64_t)(p + 1) * nt / kMeanParts);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (v < nvec) {
        for (int32_t t0 = ta; t0 < tz; t0 += kMeanUnroll) {
            uint4 y[kMeanUnroll];
#pragma unroll
            for (int u = 0; u < kMeanUnroll; ++u)
                if (t0 + u < tz) y[u] = __ldcs(A + (int64_t)(t0 + u) * nvec + v);
#pragma unroll
            for (int u = 0; u < kMeanUnroll; ++u)
                if (t0 + u < tz) acc_add<BF16>(acc, y[u]);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s_part[p][e][vi] = acc[e];
    __syncthreads();
    if (p == 0 && v < nvec) {
#pragma unroll
        for (int q = 1; q < kMeanParts; ++q)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += s_part[q][e][vi];
        __stcs(out + v, acc_weigh<BF16>(acc, (float)nt));
    }
}

}  // namespace

extern "C" tdp_status tdp_cond_blend(tdp_plan_t plan, int32_t N, int32_t ncap, const void *Ycond,
                                     const int32_t *slot, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (N < 0 || ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need N >= 0 and ncap >= 1");
    if (g.B == 0 || N == 0) return tdp_ok();
    if (!Ycond || !slot || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null Ycond, slot or out");
    if (!tdp_aligned(Ycond, 16) || !tdp_aligned(out, 16) || !tdp_aligned(slot, 4))
        return tdp_fail(TDP_ERR_MISALIGNED, "Ycond and out need 16-byte, slot 4-byte alignment");
    const int32_t CV = (g.C * g.esize) >> 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    cudaError_t err;
    if (g.nt <= kStageTiles && (uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap <= 0xffffffffull) {
        const int64_t blocks = (int64_t)g.B * ((N + kTok - 1) / kTok);
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
        const size_t smem = rows_layout(g.nt).bytes;
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_cond_blend_rows_kernel<1>, (unsigned)blocks, kTokThreads, smem, s, g, N,
                                    ncap, CV, y, slot, o)
                  : tdp_launch_smem(true, tdp_cond_blend_rows_kernel<0>, (unsigned)blocks, kTokThreads, smem, s, g, N,
                                    ncap, CV, y, slot, o);
    } else {
        const int64_t warps = (int64_t)g.B * N;              // one warp per conditioning token
        const int64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
        err = g.dtype == TDP_BF16
                  ? tdp_launch(true, tdp_cond_blend_kernel<1>, (unsigned)blocks, kThreads, s, g, N, ncap, CV, y, slot, o)
                  : tdp_launch(true, tdp_cond_blend_kernel<0>, (unsigned)blocks, kThreads, s, g, N, ncap, CV, y, slot, o);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_tile_mean(tdp_plan_t plan, int64_t L, const void *A, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (L < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "L must be >= 0");
    if (g.B == 0 || L == 0) return tdp_ok();
    if (!A || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null A or out");
    if ((L * g.esize) % 16 != 0) return tdp_fail(TDP_ERR_MISALIGNED, "L * element size must be a multiple of 16");
    if (!tdp_aligned(A, 16) || !tdp_aligned(out, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "A and out must be 16-byte aligned");
    const int64_t nvec = (int64_t)g.B * L * g.esize / 16;
    const int64_t blocks = (nvec + kMeanVecs - 1) / kMeanVecs;
    if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "tile mean grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *a = reinterpret_cast<const uint4 *>(A);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    const unsigned threads = kMeanVecs * kMeanParts;
    cudaError_t err = g.dtype == TDP_BF16
                          ? tdp_launch(true, tdp_tile_mean_kernel<1>, (unsigned)blocks, threads, s, g.nt, nvec, a, o)
                          : tdp_launch(true, tdp_tile_mean_kernel<0>, (unsigned)blocks, threads, s, g.nt, nvec, a, o);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
