// tdp_cond.cu -- the two reductions over tiles besides the latent blend
// ("Tiled Data Parallelism (TDP)"):
//   tdp_cond_blend_kernel  each conditioning token's per-tile outputs averaged
//                          over the tiles that kept it ("Shared negative
//                          (reference) positions": weight 1/(tiles that kept it));
//   tdp_tile_mean_kernel   the audio latent averaged over all tiles ("What it
//                          is": audio is processed on every tile and averaged).
// Both are gather form and accumulate in fp32 in ascending tile order; no
// atomics, no scratch.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kTileUnroll = 16;   // tiles whose loads a thread keeps in flight

template <int BF16>
__device__ __forceinline__ void acc_add(float (&a)[8], const uint4 &y)
{
    const uint32_t w[4] = {y.x, y.y, y.z, y.w};
    if (BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] += tdp_bf16_lo(w[i]);
            a[2 * i + 1] += tdp_bf16_hi(w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] += __uint_as_float(w[i]);
    }
}

template <int BF16>
__device__ __forceinline__ uint4 acc_div(const float (&a)[8], float n)
{
    if (BF16)
        return make_uint4(tdp_pack_bf16x2(__fdiv_rn(a[0], n), __fdiv_rn(a[1], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[2], n), __fdiv_rn(a[3], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[4], n), __fdiv_rn(a[5], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[6], n), __fdiv_rn(a[7], n)));
    return make_uint4(__float_as_uint(__fdiv_rn(a[0], n)), __float_as_uint(__fdiv_rn(a[1], n)),
                      __float_as_uint(__fdiv_rn(a[2], n)), __float_as_uint(__fdiv_rn(a[3], n)));
}

// Warp = one conditioning token (b, k).  Per round of 32 tiles, lane l loads the
// token's slot in tile t0 + l; a ballot gives the tiles that kept it, in
// ascending order, and their rows (lanes across the channel vectors) are loaded
// up to kRowsInFlight at a time and accumulated in that order.
constexpr int kRowsInFlight = 4;

template <int BF16>
__global__ void __launch_bounds__(kThreads)
tdp_cond_blend_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV,
                      const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot, uint4 *__restrict__ out)
{
    const int32_t lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (tok >= (int64_t)g.B * N) return;                 // warp-uniform
    const int32_t b = (int32_t)(tok / N), k = (int32_t)(tok - (int64_t)b * N);
    for (int32_t cv0 = 0; cv0 < CV; cv0 += 32) {
        const int32_t cv = cv0 + lane;
        const bool act = cv < CV;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int32_t n = 0;
        for (int32_t t0 = 0; t0 < g.nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < g.nt ? __ldg(slot + ((int64_t)t * g.B + b) * N + k) : -1;
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
                n += got;
            }
        }
        if (act) __stcs(out + tok * CV + cv, n > 0 ? acc_div<BF16>(acc, (float)n) : make_uint4(0u, 0u, 0u, 0u));
    }
}

// Thread = output vector of out[B, L].
template <int BF16>
__global__ void __launch_bounds__(kThreads)
tdp_tile_mean_kernel(int32_t nt, int64_t nvec, const uint4 *__restrict__ A, uint4 *__restrict__ out)
{
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= nvec) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int32_t t0 = 0; t0 < nt; t0 += kTileUnroll) {
        uint4 y[kTileUnroll];
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u)
            if (t0 + u < nt) y[u] = __ldcs(A + (int64_t)(t0 + u) * nvec + v);
#pragma unroll
        for (int u = 0; u < kTileUnroll; ++u)
            if (t0 + u < nt) acc_add<BF16>(acc, y[u]);
    }
    __stcs(out + v, acc_div<BF16>(acc, (float)nt));
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
    const int64_t warps = (int64_t)g.B * N;                  // one warp per conditioning token
    const int64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
    if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    if (g.dtype == TDP_BF16)
        tdp_cond_blend_kernel<1><<<(unsigned)blocks, kThreads, 0, s>>>(g, N, ncap, CV, y, slot, o);
    else
        tdp_cond_blend_kernel<0><<<(unsigned)blocks, kThreads, 0, s>>>(g, N, ncap, CV, y, slot, o);
    const cudaError_t err = cudaGetLastError();
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
    const int64_t blocks = (nvec + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "tile mean grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *a = reinterpret_cast<const uint4 *>(A);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    if (g.dtype == TDP_BF16)
        tdp_tile_mean_kernel<1><<<(unsigned)blocks, kThreads, 0, s>>>(g.nt, nvec, a, o);
    else
        tdp_tile_mean_kernel<0><<<(unsigned)blocks, kThreads, 0, s>>>(g.nt, nvec, a, o);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
