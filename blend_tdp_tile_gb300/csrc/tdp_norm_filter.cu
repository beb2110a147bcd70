// tdp_norm_filter.cu -- per-tile conditioning-token filter and normalisation
// ("Tiled Data Parallelism (TDP)", sections "Shared negative (reference)
// positions" and "Position normalization").
//
// No scratch memory, no atomics, no block waits on another.  Two forms:
//
// Up to kOneChunk tokens (one chunk per (tile, batch item)): one launch,
// tdp_filter_kernel, of two kinds of 512-thread block: a filter block per (tile, batch
// item), tdp_filter.cuh's tb_block (keep test, keep bytes, stable compaction, -1 padding,
// count), and count blocks (the tiles that keep each token).
//
// More tokens: two launches, both over (tile, batch item, chunk of 4096 tokens) blocks so
// that the work spreads over the whole GPU even with few tiles (the keep output carries
// what the second launch needs):
//   1. tdp_keep_kernel: every thread tests 16 tokens of its chunk, 256 apart
//      (coalesced), against the tile's position extent [mn, mx) and writes the
//      keep byte.  Extra blocks count, for each token, the tiles that keep it
//      (the 1/(tiles that kept it) weight's denominator), re-running the same
//      test against tile bounds staged in shared memory.
//   2. tdp_compact_kernel: a block sums the keep bytes of its (tile, batch
//      item) before its chunk and in all (keep bytes are 0/1, so a popcount
//      per word counts them), places its chunk's kept tokens in ascending order
//      with one scan of a (sub-chunk, warp) count table, writes idx, the
//      shifted intervals and the slots, and pads its own range of idx with -1.
#include "tdp.h"
#include "tdp_filter.cuh"
#include "tdp_internal.h"

namespace {

using namespace tdp_filt;

constexpr int kOneThreads = 512;                      // threads of the one-launch form's blocks
constexpr int kOneChunk = kOneThreads * kSub;         // most tokens the one-launch form takes

// Blocks [0, nfilt): filter blocks (tb = t*B + b); [nfilt, nfilt + ncount): count blocks.
__global__ void __launch_bounds__(kOneThreads)
tdp_filter_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ K, int32_t N,
                  const int32_t *__restrict__ mn, const int32_t *__restrict__ mx, int32_t normalize,
                  uint8_t *__restrict__ keep, int32_t *__restrict__ idx, int32_t *__restrict__ count,
                  int32_t *__restrict__ kcount, int2 *__restrict__ Kout, int32_t *__restrict__ slot, int32_t nfilt)
{
    __shared__ union {
        compact_smem_t<kOneThreads> compact;
        kcount_smem_t<kOneThreads> kc;
    } sm;
    // No early trigger: the next kernel launches as these latency-bound blocks exit.
    tdp_pdl_wait();
    if ((int32_t)blockIdx.x < nfilt)
        tb_block<kOneThreads>(g, K, N, mn, mx, normalize, blockIdx.x, keep, idx, count, Kout, slot, sm.compact);
    else
        kcount_block<kOneThreads>(g, K, N, mn, mx, kcount, (int32_t)blockIdx.x - nfilt, sm.kc);
}

__global__ void __launch_bounds__(kThreads)
tdp_keep_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ K, int32_t N, int32_t nchunk,
                const int32_t *__restrict__ mn, const int32_t *__restrict__ mx, uint8_t *__restrict__ keep,
                int32_t *__restrict__ kcount)
{
    __shared__ kcount_smem sm;
    // No early trigger here or in tdp_compact_kernel: the next kernel launches as these
    // blocks exit.  Blocks of the next kernel waiting beside these latency-bound ones
    // slowed them more than the early launch saved.
    tdp_pdl_wait();
    const int64_t nkeep = (int64_t)g.nt * g.B * nchunk;
    if ((int64_t)blockIdx.x < nkeep) {
        // ---- keep bytes of (t, b), chunk c
        const int64_t tb = blockIdx.x / nchunk;
        const int32_t c = (int32_t)(blockIdx.x - tb * nchunk);
        const int32_t b = (int32_t)(tb % g.B);
        const int2 *Kb = K + (int64_t)b * 3 * N;
        int32_t lo[3], hi[3];
        load_bounds(mn, mx, tb, lo, hi);
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
            const int32_t k = c * kChunk + j * kThreads + threadIdx.x;
            if (k < N) {
                const int2 kv[3] = {__ldg(Kb + k), __ldg(Kb + (int64_t)N + k), __ldg(Kb + 2 * (int64_t)N + k)};
                keep[tb * N + k] = keeps(kv, lo, hi) ? 1 : 0;
            }
        }
        return;
    }
    kcount_block(g, K, N, mn, mx, kcount, (int32_t)(blockIdx.x - nkeep), sm);
}

// Sum over the block of two values (every thread calls it).
__device__ __forceinline__ void block_sum2(int32_t &x, int32_t &y, int32_t (*s)[2])
{
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = __reduce_add_sync(0xffffffffu, x);
    y = __reduce_add_sync(0xffffffffu, y);
    if (lane == 0) {
        s[warp][0] = x;
        s[warp][1] = y;
    }
    __syncthreads();
    x = 0;
    y = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        x += s[w][0];
        y += s[w][1];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
tdp_compact_kernel(const __grid_constant__ tdp_geom g, const int2 *__restrict__ K, int32_t N, int32_t nchunk,
                   const int32_t *__restrict__ mn, int32_t normalize, const uint8_t *__restrict__ keep,
                   int32_t vec16, int32_t *__restrict__ idx, int32_t *__restrict__ count,
                   int2 *__restrict__ Kout, int32_t *__restrict__ slot)
{
    __shared__ compact_smem sm;
    __shared__ int32_t s_sum[kWarps][2];
    tdp_pdl_wait();
    const int64_t tb = blockIdx.x / nchunk;
    const int32_t c = (int32_t)(blockIdx.x - tb * nchunk);
    const int32_t b = (int32_t)(tb % g.B);
    const uint8_t *krow = keep + tb * N;
    const int32_t k0 = c * kChunk;

    // ---- kept tokens of (t, b) before this chunk and in all
    int32_t before = 0, total = 0;
    if (vec16) {          // keep 16-byte aligned and N % 16 == 0 (checked on the host): 16 bytes per load
        const uint4 *q = reinterpret_cast<const uint4 *>(krow);
        for (int32_t i = threadIdx.x; i < N / 16; i += blockDim.x) {
            const uint4 v = __ldg(q + i);
            const int32_t n = __popc(v.x) + __popc(v.y) + __popc(v.z) + __popc(v.w);
            total += n;
            before += i * 16 < k0 ? n : 0;
        }
    } else {
        for (int32_t i = threadIdx.x; i < N; i += blockDim.x) {
            const int32_t n = __ldg(krow + i);
            total += n;
            before += i < k0 ? n : 0;
        }
    }
    block_sum2(before, total, s_sum);

    // ---- this chunk: ballots per (sub-chunk, warp), offsets from one scan
    uint32_t ballots[kSub];
#pragma unroll
    for (int j = 0; j < kSub; ++j) {
        const int32_t k = k0 + j * kThreads + threadIdx.x;
        ballots[j] = __ballot_sync(0xffffffffu, k < N && __ldg(krow + k) != 0);
    }
    chunk_offsets(ballots, before, sm);
    int32_t shift[3] = {0, 0, 0};
    if (normalize) {
#pragma unroll
        for (int d = 0; d < 3; ++d) shift[d] = __ldg(mn + tb * 3 + d);
    }
    chunk_write(K + (int64_t)b * 3 * N, N, tb, k0, ballots, shift, sm, idx, Kout, slot);
    // ---- idx past the total count: -1, over this chunk's range of positions
    for (int32_t p = max(total, k0) + threadIdx.x; p < min(N, k0 + kChunk); p += blockDim.x) idx[tb * N + p] = -1;
    if (c == 0 && threadIdx.x == 0) count[tb] = total;
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
    using namespace tdp_filt;
    const int32_t nchunk = N > 0 ? (N + kChunk - 1) / kChunk : 1;
    const int64_t nkeep = (int64_t)g.nt * g.B * nchunk;
    const int64_t blocks1 = nkeep + (int64_t)g.B * ((N + kCountTok - 1) / kCountTok);
    if (blocks1 > 0x7fffffffLL || (int64_t)g.B * N * g.nt > ((int64_t)1 << 56))
        return tdp_fail(TDP_ERR_TOO_LARGE, "filter grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int2 *k2 = reinterpret_cast<const int2 *>(K);
    cudaError_t err = cudaSuccess;
    if (N <= kOneChunk) {
        const int64_t ncount = (int64_t)g.B * ((N + kCountTok - 1) / kCountTok);
        err = tdp_launch(true, tdp_filter_kernel, (unsigned)(g.nt * (int64_t)g.B + ncount), kOneThreads, s, g, k2, N,
                         mn, mx, normalize, keep, idx, count, kcount, reinterpret_cast<int2 *>(Kout), slot,
                         (int32_t)(g.nt * (int64_t)g.B));
        if (err == cudaSuccess) err = cudaGetLastError();
        if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
        return tdp_ok();
    }
    if (N > 0)
        err = tdp_launch(true, tdp_keep_kernel, (unsigned)blocks1, kThreads, s, g, k2, N, nchunk, mn, mx, keep,
                         kcount);
    // every row keep + tb*N is then 16-byte aligned too
    const int32_t vec16 = N % 16 == 0 && tdp_aligned(keep, 16) ? 1 : 0;
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_compact_kernel, (unsigned)nkeep, kThreads, s, g, k2, N, nchunk, mn, normalize,
                         static_cast<const uint8_t *>(keep), vec16, idx, count, reinterpret_cast<int2 *>(Kout),
                         slot);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
