// tdp_norm_filter.cu -- per-tile conditioning-token filter and normalisation
// ("Tiled Data Parallelism (TDP)", sections "Shared negative (reference)
// positions" and "Position normalization").
//
// One launch.  Blocks [0, n_tiles*B) each own one (tile, batch item): they
// test every conditioning token against the tile's position extent
// [mn, mx), compact the kept ones in ascending token order (warp ballots and
// a block-wide scan of the warp counts, no atomics) and write them shifted by
// mn.  The remaining blocks own (batch item, token) pairs and count the tiles
// that keep each token (the 1/(tiles that kept it) weight's denominator),
// re-running the same keep test, so no block waits on another.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kFilterThreads = 512;

// Keep rule: the interval overlaps the tile's extent in all three dimensions
// ([max(s, mn), min(e, mx)) non-empty), or its time start is negative.
__device__ __forceinline__ bool tdp_keeps(const int2 (&k)[3], const int32_t (&lo)[3], const int32_t (&hi)[3])
{
    bool inside = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) inside &= max(k[d].x, lo[d]) < min(k[d].y, hi[d]);
    return inside || k[0].x < 0;
}

__global__ void __launch_bounds__(kFilterThreads)
tdp_filter_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ K, int32_t N,
                  const int32_t *__restrict__ mn, const int32_t *__restrict__ mx, int32_t normalize,
                  uint8_t *__restrict__ keep, int32_t *__restrict__ idx, int32_t *__restrict__ count,
                  int32_t *__restrict__ kcount, int2 *__restrict__ Kout)
{
    const int32_t ntb = g.nt * g.B;
    if ((int32_t)blockIdx.x >= ntb) {
        // ---- kcount[b, k] = number of tiles keeping token k of item b
        const int64_t gid = (int64_t)(blockIdx.x - ntb) * blockDim.x + threadIdx.x;
        if (gid >= (int64_t)g.B * N) return;
        const int32_t b = (int32_t)(gid / N), k = (int32_t)(gid % N);
        int2 kv[3];
#pragma unroll
        for (int d = 0; d < 3; ++d) kv[d] = __ldg(K + ((int64_t)b * 3 + d) * N + k);
        int32_t cnt = 0;
        for (int32_t t = 0; t < g.nt; ++t) {
            const int64_t r = ((int64_t)t * g.B + b) * 3;
            int32_t lo[3], hi[3];
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                lo[d] = __ldg(mn + r + d);
                hi[d] = __ldg(mx + r + d);
            }
            cnt += tdp_keeps(kv, lo, hi) ? 1 : 0;
        }
        kcount[gid] = cnt;
        return;
    }

    // ---- compaction for (t, b) = blockIdx.x / B, blockIdx.x % B
    const int32_t tb = blockIdx.x;
    const int32_t b = tb % g.B;
    int32_t lo[3], hi[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        lo[d] = __ldg(mn + (int64_t)tb * 3 + d);
        hi[d] = __ldg(mx + (int64_t)tb * 3 + d);
    }
    __shared__ int32_t s_warp[kFilterThreads / 32];
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t nwarp = blockDim.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    int32_t base = 0;   // kept tokens before this chunk (uniform)
    for (int32_t k0 = 0; k0 < N; k0 += blockDim.x) {
        const int32_t k = k0 + threadIdx.x;
        int2 kv[3] = {make_int2(0, 0), make_int2(0, 0), make_int2(0, 0)};
        bool kept = false;
        if (k < N) {
#pragma unroll
            for (int d = 0; d < 3; ++d) kv[d] = __ldg(K + ((int64_t)b * 3 + d) * N + k);
            kept = tdp_keeps(kv, lo, hi);
            keep[(int64_t)tb * N + k] = kept ? 1 : 0;
        }
        const uint32_t ballot = __ballot_sync(0xffffffffu, kept);
        if (lane == 0) s_warp[warp] = __popc(ballot);
        __syncthreads();
        int32_t before = 0, total = 0;
        for (int32_t w = 0; w < nwarp; ++w) {
            const int32_t c = s_warp[w];
            before += w < warp ? c : 0;
            total += c;
        }
        if (kept) {
            const int32_t pos = base + before + __popc(ballot & lt_mask);
            idx[(int64_t)tb * N + pos] = k;
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                int2 o = kv[d];
                if (normalize) {
                    o.x = (int32_t)((uint32_t)o.x - (uint32_t)lo[d]);
                    o.y = (int32_t)((uint32_t)o.y - (uint32_t)lo[d]);
                }
                Kout[((int64_t)tb * 3 + d) * N + pos] = o;
            }
        }
        base += total;
        __syncthreads();   // s_warp is rewritten by the next chunk
    }
    for (int32_t k = base + threadIdx.x; k < N; k += blockDim.x) idx[(int64_t)tb * N + k] = -1;
    if (threadIdx.x == 0) count[tb] = base;
}

}  // namespace

extern "C" tdp_status tdp_norm_filter(tdp_plan_t plan, const int32_t *K, int32_t N,
                                      const int32_t *mn, const int32_t *mx, int32_t normalize,
                                      uint8_t *keep, int32_t *idx, int32_t *count, int32_t *kcount,
                                      int32_t *Kout, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (N < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "N must be >= 0");
    if (g.B == 0) return tdp_ok();
    if (!mn || !mx || !count) return tdp_fail(TDP_ERR_INVALID_ARG, "null mn, mx or count");
    if (N > 0 && (!K || !keep || !idx || !kcount || !Kout))
        return tdp_fail(TDP_ERR_INVALID_ARG, "null K, keep, idx, kcount or Kout");
    if (!tdp_aligned(mn, 4) || !tdp_aligned(mx, 4) || !tdp_aligned(count, 4) ||
        (N > 0 && (!tdp_aligned(K, 8) || !tdp_aligned(Kout, 8) || !tdp_aligned(idx, 4) ||
                   !tdp_aligned(kcount, 4))))
        return tdp_fail(TDP_ERR_MISALIGNED, "K, Kout need 8-byte and int32 buffers 4-byte alignment");
    const int64_t ntb = (int64_t)g.nt * g.B;
    // both block kinds share one launch: n_tiles*B compaction blocks, then count blocks
    const int64_t blocks = ntb + ((int64_t)g.B * N + kFilterThreads - 1) / kFilterThreads;
    if (blocks > 0x7fffffffLL || (int64_t)g.B * N * g.nt > ((int64_t)1 << 56))
        return tdp_fail(TDP_ERR_TOO_LARGE, "filter grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tdp_filter_kernel<<<(unsigned)blocks, kFilterThreads, 0, s>>>(
        g, reinterpret_cast<const int2 *>(K), N, mn, mx, normalize, keep, idx, count, kcount,
        reinterpret_cast<int2 *>(Kout));
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
