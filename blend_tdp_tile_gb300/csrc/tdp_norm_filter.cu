// tdp_norm_filter.cu -- per-tile conditioning-token filter and normalisation
// ("Tiled Data Parallelism (TDP)", sections "Shared negative (reference)
// positions" and "Position normalization").
//
// One launch, one block of 1024 threads per (tile, batch item):
//   1. compaction, in passes of 16384 tokens.  Warp w tests tokens
//      j*1024 + w*32 + lane for j = 0..15 (every load and store coalesced) and
//      keeps the 16 ballots; the 16 x 32 table of per-(j, warp) counts is
//      scanned once in (j, warp) order, so token k's slot is its table offset
//      plus its rank within its ballot: ascending order, no atomics.  Kept
//      tokens are written shifted by mn, and (optionally) every token's slot in
//      the kept list (or -1).
//   2. keep counts: the B*n_tiles blocks split each batch item's tokens into
//      n_tiles slices; a block counts, for each token of its slice, the tiles
//      that keep it (the 1/(tiles that kept it) weight's denominator) by
//      re-running the same keep test against tile bounds staged in shared
//      memory, the tiles split over 8 thread groups.
// No block waits on another.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kFilterThreads = 1024;
constexpr int kWarps = kFilterThreads / 32;
constexpr int kSub = 16;                          // sub-chunks of 1024 tokens per pass
constexpr int kPass = kFilterThreads * kSub;
constexpr int kCountTok = 128;                    // tokens per keep-count round
constexpr int kCountGroups = kFilterThreads / kCountTok;
constexpr int kTileStage = 1024;                  // tile bounds staged in shared memory at once

// Keep rule: the interval overlaps the tile's extent in all three dimensions
// ([max(s, mn), min(e, mx)) non-empty), or its time start is negative.
__device__ __forceinline__ bool tdp_keeps(const int2 (&k)[3], const int32_t (&lo)[3], const int32_t (&hi)[3])
{
    bool inside = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) inside &= max(k[d].x, lo[d]) < min(k[d].y, hi[d]);
    return inside || k[0].x < 0;
}

__global__ void __launch_bounds__(kFilterThreads, 1)
tdp_filter_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ K, int32_t N,
                  const int32_t *__restrict__ mn, const int32_t *__restrict__ mx, int32_t normalize,
                  uint8_t *__restrict__ keep, int32_t *__restrict__ idx, int32_t *__restrict__ count,
                  int32_t *__restrict__ kcount, int2 *__restrict__ Kout, int32_t *__restrict__ slot)
{
    __shared__ int32_t s_off[kSub][kWarps];       // per (sub-chunk, warp): kept count, then offset
    __shared__ int32_t s_total;
    __shared__ int32_t s_lo[kTileStage][3], s_hi[kTileStage][3];
    __shared__ int32_t s_cnt[kCountGroups][kCountTok];
    const int32_t tb = blockIdx.x;                 // t*B + b
    const int32_t t = tb / g.B, b = tb % g.B;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int2 *Kb = K + (int64_t)b * 3 * N;

    // ---- 1. compaction of (t, b)
    int32_t lo[3], hi[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        lo[d] = __ldg(mn + (int64_t)tb * 3 + d);
        hi[d] = __ldg(mx + (int64_t)tb * 3 + d);
    }
    int32_t base = 0;   // kept tokens before this pass (uniform)
    for (int32_t k0 = 0; k0 < N; k0 += kPass) {
        uint32_t ballots[kSub];
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
            const int32_t k = k0 + j * kFilterThreads + warp * 32 + lane;
            bool kept = false;
            if (k < N) {
                const int2 kv[3] = {__ldg(Kb + k), __ldg(Kb + (int64_t)N + k), __ldg(Kb + 2 * (int64_t)N + k)};
                kept = tdp_keeps(kv, lo, hi);
                keep[(int64_t)tb * N + k] = kept ? 1 : 0;
            }
            ballots[j] = __ballot_sync(0xffffffffu, kept);
        }
        if (lane < kSub) {
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < kSub; ++j) mine = lane == j ? ballots[j] : mine;
            s_off[lane][warp] = __popc(mine);
        }
        __syncthreads();
        if (warp == 0) {
            // exclusive scan of the kSub*kWarps counts in (j, warp) order: lane l owns row j = l
            int32_t row[kWarps];
            int32_t sum = 0;
            if (lane < kSub) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    row[w] = s_off[lane][w];
                    sum += row[w];
                }
            }
            int32_t incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            if (lane < kSub) {
                int32_t run = incl - sum;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    s_off[lane][w] = run;
                    run += row[w];
                }
            }
            if (lane == 31) s_total = incl;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
            const int32_t kj = k0 + j * kFilterThreads + warp * 32 + lane;
            const bool kept = (ballots[j] >> lane) & 1u;
            if (slot && kj < N)
                slot[(int64_t)tb * N + kj] = kept ? base + s_off[j][warp] + __popc(ballots[j] & lt_mask) : -1;
            if (kept) {
                const int32_t k = kj;
                const int32_t pos = base + s_off[j][warp] + __popc(ballots[j] & lt_mask);
                idx[(int64_t)tb * N + pos] = k;
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    int2 o = __ldg(Kb + (int64_t)d * N + k);
                    if (normalize) {
                        o.x = (int32_t)((uint32_t)o.x - (uint32_t)lo[d]);
                        o.y = (int32_t)((uint32_t)o.y - (uint32_t)lo[d]);
                    }
                    Kout[((int64_t)tb * 3 + d) * N + pos] = o;
                }
            }
        }
        base += s_total;
        __syncthreads();   // s_off and s_total are rewritten by the next pass
    }
    for (int32_t k = base + threadIdx.x; k < N; k += blockDim.x) idx[(int64_t)tb * N + k] = -1;
    if (threadIdx.x == 0) count[tb] = base;

    // ---- 2. keep counts of this block's slice of item b's tokens
    const int32_t per = (N + g.nt - 1) / g.nt;
    const int32_t ks0 = min(N, t * per), ks1 = min(N, ks0 + per);
    if (ks0 >= ks1) return;   // uniform over the block
    const int32_t tok = threadIdx.x % kCountTok, grp = threadIdx.x / kCountTok;
    for (int32_t kc = ks0; kc < ks1; kc += kCountTok) {
        const int32_t k = kc + tok;
        int2 kv[3] = {make_int2(0, 0), make_int2(0, 0), make_int2(0, 0)};
        if (k < ks1) {
#pragma unroll
            for (int d = 0; d < 3; ++d) kv[d] = __ldg(Kb + (int64_t)d * N + k);
        }
        int32_t cnt = 0;
        for (int32_t u0 = 0; u0 < g.nt; u0 += kTileStage) {
            const int32_t un = min(kTileStage, g.nt - u0);
            __syncthreads();   // previous readers of s_lo / s_hi are done
            for (int32_t i = threadIdx.x; i < un * 3; i += blockDim.x) {
                const int32_t u = i / 3, d = i - u * 3;
                const int64_t r = ((int64_t)(u0 + u) * g.B + b) * 3 + d;
                s_lo[u][d] = __ldg(mn + r);
                s_hi[u][d] = __ldg(mx + r);
            }
            __syncthreads();
            for (int32_t u = grp; u < un; u += kCountGroups) {     // warp-uniform: shared broadcast
                const int32_t a[3] = {s_lo[u][0], s_lo[u][1], s_lo[u][2]};
                const int32_t z[3] = {s_hi[u][0], s_hi[u][1], s_hi[u][2]};
                cnt += tdp_keeps(kv, a, z) ? 1 : 0;
            }
        }
        s_cnt[grp][tok] = cnt;
        __syncthreads();
        if (grp == 0 && k < ks1) {
            int32_t sum = 0;
#pragma unroll
            for (int i = 0; i < kCountGroups; ++i) sum += s_cnt[i][tok];
            kcount[(int64_t)b * N + k] = sum;
        }
    }
}

}  // namespace

extern "C" tdp_status tdp_norm_filter(tdp_plan_t plan, const int32_t *K, int32_t N,
                                      const int32_t *mn, const int32_t *mx, int32_t normalize,
                                      uint8_t *keep, int32_t *idx, int32_t *count, int32_t *kcount,
                                      int32_t *Kout, int32_t *slot, tdp_stream_t stream)
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
                   !tdp_aligned(kcount, 4) || !tdp_aligned(slot, 4))))
        return tdp_fail(TDP_ERR_MISALIGNED, "K, Kout need 8-byte and int32 buffers 4-byte alignment");
    const int64_t blocks = (int64_t)g.nt * g.B;    // one block per (tile, batch item)
    if (blocks > 0x7fffffffLL || (int64_t)g.B * N * g.nt > ((int64_t)1 << 56))
        return tdp_fail(TDP_ERR_TOO_LARGE, "filter grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tdp_filter_kernel<<<(unsigned)blocks, kFilterThreads, 0, s>>>(
        g, reinterpret_cast<const int2 *>(K), N, mn, mx, normalize, keep, idx, count, kcount,
        reinterpret_cast<int2 *>(Kout), slot);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
