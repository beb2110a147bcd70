// tdp_filter.cuh -- device pieces of the per-tile conditioning-token filter
// ("Tiled Data Parallelism (TDP)", sections "Shared negative (reference)
// positions" and "Position normalization"), shared by the two-launch filter
// (tdp_norm_filter) and the fused split + filter launch (tdp_split_filter).
//
// Keep rule for token k of batch item b and tile t, in global coordinates:
// its interval overlaps the tile's position extent [mn, mx) in all three
// dimensions, or its time start is negative.  Kept tokens are listed in
// ascending k (stable compaction), shifted by the tile's mn when normalising.
#pragma once

#include "tdp_device.cuh"

namespace tdp_filt {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSub = 16;                          // tokens per thread and chunk
constexpr int kChunk = kThreads * kSub;           // tokens per chunk
constexpr int kCountTok = 64;                     // tokens per keep-count block
constexpr int kTileStage = 1024;                  // tile bounds staged in shared memory at once

__device__ __forceinline__ bool keeps(const int2 (&k)[3], const int32_t (&lo)[3], const int32_t (&hi)[3])
{
    bool inside = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) inside &= max(k[d].x, lo[d]) < min(k[d].y, hi[d]);
    return inside || k[0].x < 0;
}

__device__ __forceinline__ void load_bounds(const int32_t *mn, const int32_t *mx, int64_t tb, int32_t (&lo)[3],
                                            int32_t (&hi)[3])
{
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        lo[d] = __ldg(mn + tb * 3 + d);
        hi[d] = __ldg(mx + tb * 3 + d);
    }
}

// ---- kcount[b, k] for the kCountTok tokens of block `blk` (blocks are (b, token
// range) in b-major order), by a block of T threads: thread (group, token) tests tiles
// t = group mod T / kCountTok against bounds staged in shared memory; the groups' counts
// are summed.
template <int T>
struct kcount_smem_t {
    int32_t lo[kTileStage][3], hi[kTileStage][3];
    int32_t cnt[T / kCountTok][kCountTok];
};
using kcount_smem = kcount_smem_t<kThreads>;

template <int T = kThreads>
__device__ __forceinline__ void kcount_block(const tdp_geom &g, const int2 *K, int32_t N, const int32_t *mn,
                                             const int32_t *mx, int32_t *kcount, int32_t blk, kcount_smem_t<T> &sm)
{
    constexpr int kCountGroups = T / kCountTok;
    const int32_t nkb = (N + kCountTok - 1) / kCountTok;
    const int32_t b = blk / nkb;
    const int32_t tok = threadIdx.x % kCountTok, grp = threadIdx.x / kCountTok;
    const int32_t k = (blk - b * nkb) * kCountTok + tok;
    const int2 *Kb = K + (int64_t)b * 3 * N;
    int2 kv[3] = {make_int2(0, 0), make_int2(0, 0), make_int2(0, 0)};
    if (k < N) {
#pragma unroll
        for (int d = 0; d < 3; ++d) kv[d] = __ldg(Kb + (int64_t)d * N + k);
    }
    int32_t cnt = 0;
    for (int32_t u0 = 0; u0 < g.nt; u0 += kTileStage) {
        const int32_t un = min(kTileStage, g.nt - u0);
        __syncthreads();   // previous readers of lo / hi are done
        for (int32_t i = threadIdx.x; i < un * 3; i += blockDim.x) {
            const int32_t u = i / 3, d = i - u * 3;
            const int64_t r = ((int64_t)(u0 + u) * g.B + b) * 3 + d;
            sm.lo[u][d] = __ldg(mn + r);
            sm.hi[u][d] = __ldg(mx + r);
        }
        __syncthreads();
        for (int32_t u = grp; u < un; u += kCountGroups) {        // warp-uniform: shared broadcast
            const int32_t a[3] = {sm.lo[u][0], sm.lo[u][1], sm.lo[u][2]};
            const int32_t z[3] = {sm.hi[u][0], sm.hi[u][1], sm.hi[u][2]};
            cnt += keeps(kv, a, z) ? 1 : 0;
        }
    }
    sm.cnt[grp][tok] = cnt;
    __syncthreads();
    if (grp == 0 && k < N) {
        int32_t sum = 0;
#pragma unroll
        for (int i = 0; i < kCountGroups; ++i) sum += sm.cnt[i][tok];
        kcount[(int64_t)b * N + k] = sum;
    }
}

// ---- compaction of one chunk of T * kSub tokens by a block of T threads.  Thread
// (warp w, lane l) owns tokens k0 + j*T + w*32 + l, j < kSub; ballots[j] are its warp's
// keep ballots.  Positions follow (j, w, l) order, i.e. ascending k.
template <int T>
struct compact_smem_t {
    int32_t off[kSub][T / 32];
    int32_t total;
};
using compact_smem = compact_smem_t<kThreads>;

// sm.off[j][w] = base + kept tokens of the chunk before sub-chunk j of warp w;
// returns the chunk's kept count.  Every thread calls it; ends with a barrier.
template <int T = kThreads>
__device__ __forceinline__ int32_t chunk_offsets(const uint32_t (&ballots)[kSub], int32_t base, compact_smem_t<T> &sm)
{
    constexpr int kWarps = T / 32;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane < kSub) {
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kSub; ++j) mine = lane == j ? ballots[j] : mine;
        sm.off[lane][warp] = __popc(mine);
    }
    __syncthreads();
    if (warp == 0) {
        // lane l < kSub owns row j = l of the (sub-chunk, warp) count table
        int32_t row[kWarps];
        int32_t sum = 0;
        if (lane < kSub) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                row[w] = sm.off[lane][w];
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
            int32_t run = base + incl - sum;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                sm.off[lane][w] = run;
                run += row[w];
            }
        }
        if (lane == 31) sm.total = incl;      // lanes >= kSub add nothing
    }
    __syncthreads();
    return sm.total;
}

// Write slot / idx / Kout for one chunk whose offsets chunk_offsets() filled.
template <int T = kThreads>
__device__ __forceinline__ void chunk_write(const int2 *Kb, int32_t N, int64_t tb, int32_t k0,
                                            const uint32_t (&ballots)[kSub], const int32_t (&shift)[3],
                                            const compact_smem_t<T> &sm, int32_t *idx, int2 *Kout, int32_t *slot)
{
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kSub; ++j) {
        const int32_t k = k0 + j * T + threadIdx.x;
        const bool kept = (ballots[j] >> lane) & 1u;
        const int32_t pos = sm.off[j][warp] + __popc(ballots[j] & lt_mask);
        if (slot && k < N) slot[tb * N + k] = kept ? pos : -1;
        if (kept) {
            idx[tb * N + pos] = k;
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                int2 o = __ldg(Kb + (int64_t)d * N + k);
                o.x = (int32_t)((uint32_t)o.x - (uint32_t)shift[d]);
                o.y = (int32_t)((uint32_t)o.y - (uint32_t)shift[d]);
                Kout[(tb * 3 + d) * N + pos] = o;
            }
        }
    }
}

// ---- the whole filter of one (tile, batch item) row tb = t*B + b in one block of T
// threads: keep test, keep bytes, stable compaction chunk by chunk (T * kSub tokens
// each) with a running base, -1 padding of idx and the count.
template <int T = kThreads>
__device__ __forceinline__ void tb_block(const tdp_geom &g, const int2 *K, int32_t N, const int32_t *mn,
                                         const int32_t *mx, int32_t normalize, int64_t tb, uint8_t *keep,
                                         int32_t *idx, int32_t *count, int2 *Kout, int32_t *slot,
                                         compact_smem_t<T> &sm)
{
    const int32_t b = (int32_t)(tb % g.B);
    const int2 *Kb = K + (int64_t)b * 3 * N;
    int32_t lo[3], hi[3];
    load_bounds(mn, mx, tb, lo, hi);
    const int32_t shift[3] = {normalize ? lo[0] : 0, normalize ? lo[1] : 0, normalize ? lo[2] : 0};
    int32_t run = 0;
    for (int32_t k0 = 0; k0 < N; k0 += T * kSub) {
        uint32_t ballots[kSub];
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
            const int32_t k = k0 + j * T + threadIdx.x;
            bool kept = false;
            if (k < N) {
                const int2 kv[3] = {__ldg(Kb + k), __ldg(Kb + (int64_t)N + k), __ldg(Kb + 2 * (int64_t)N + k)};
                kept = keeps(kv, lo, hi);
                keep[tb * N + k] = kept ? 1 : 0;
            }
            ballots[j] = __ballot_sync(0xffffffffu, kept);
        }
        const int32_t tot = chunk_offsets<T>(ballots, run, sm);
        chunk_write<T>(Kb, N, tb, k0, ballots, shift, sm, idx, Kout, slot);
        run += tot;
        __syncthreads();                      // the next chunk rewrites sm.off / sm.total
    }
    for (int32_t p = run + threadIdx.x; p < N; p += blockDim.x) idx[tb * N + p] = -1;
    if (threadIdx.x == 0) count[tb] = run;
}

}  // namespace tdp_filt
