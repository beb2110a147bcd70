// tdp_cond_rec.cu -- the conditioning-token output reduction in two calls, for callers
// whose conditioning tokens, and so the filter's slots, stay the same from call to call
// ("Tiled Data Parallelism (TDP)", section "Shared negative (reference) positions": a token
// kept by several tiles has blend weight 1/(number of tiles that kept it)):
//   tdp_cond_records        once: every token block's record (tdp_cond_rows.cuh: its rows of
//                           Ycond, the rows per token and the tiles that kept each token),
//                           stored in launch order, the blocks with the most rows first;
//   tdp_cond_blend_records  each call: the outputs from the records, bit for bit those of
//                           tdp_cond_blend.
// The per-call kernel reads its block's record in one trip instead of staging the slots and
// building the lists, and the blocks that take longest start first.
//
// tdp_cond_records runs three kernels: tdp_cond_count_kernel (a block's stored rows, from
// the slots), tdp_cond_order_kernel (one block: each token block's launch position, a stable
// sort by the number of ring stages its rows fill, most first) and tdp_cond_record_kernel
// (the records, written at their positions).
#include "tdp.h"
#include "tdp_cond_rows.cuh"
#include "tdp_internal.h"

namespace {

using namespace tdp_cr;

constexpr int kOrderThreads = 1024;
constexpr int kClasses = 8;        // launch classes: ring stages the rows fill, 7 or more in class 7

__device__ __forceinline__ int32_t launch_class(int32_t R)
{
    const int32_t u = (R + kChunkRows - 1) / kChunkRows;
    return u < kClasses - 1 ? u : kClasses - 1;
}

// pos[blk] = rows stored for token block blk.
__global__ void __launch_bounds__(kTokThreads, kTokMinBlocks)
tdp_cond_count_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, const int32_t *__restrict__ slot,
                      int32_t *__restrict__ pos)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    int32_t *rec = reinterpret_cast<int32_t *>(dsm + rows_layout(g.nt).rec);
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t blk = blockIdx.x;
    const int32_t nkb = (N + kTok - 1) / kTok;
    const int32_t b = blk / nkb, k0 = (blk - b * nkb) * kTok;
    const tok_rows tr = rows_from_slots(g, N, ncap, slot, blk, b, k0, dsm, rec);
    if (threadIdx.x == 0) pos[blk] = tr.R;
}

// One block: pos[i] (rows of token block i) becomes block i's launch position.  Classes in
// descending order, blocks of a class in ascending order; every position in [0, G) once.
__global__ void __launch_bounds__(kOrderThreads)
tdp_cond_order_kernel(int32_t G, int32_t *__restrict__ pos)
{
    constexpr int kW = kOrderThreads / 32;
    __shared__ int32_t s_cnt[kClasses], s_carry[kClasses];
    __shared__ int32_t s_wc[kW][kClasses];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < kClasses) s_cnt[threadIdx.x] = 0;
    __syncthreads();
    for (int32_t i = threadIdx.x; i < G; i += kOrderThreads) atomicAdd(&s_cnt[launch_class(pos[i])], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t run = 0;
        for (int c = kClasses - 1; c >= 0; --c) {
            s_carry[c] = run;
            run += s_cnt[c];
        }
    }
    __syncthreads();
    for (int32_t i0 = 0; i0 < G; i0 += kOrderThreads) {
        const int32_t i = i0 + (int32_t)threadIdx.x;
        const int32_t c = i < G ? launch_class(pos[i]) : -1;
        uint32_t mine = 0;
#pragma unroll
        for (int cc = 0; cc < kClasses; ++cc) {
            const uint32_t m = __ballot_sync(0xffffffffu, c == cc);
            if (c == cc) mine = m;
            if (lane == 0) s_wc[warp][cc] = __popc(m);
        }
        __syncthreads();
        if (threadIdx.x < kClasses) {                     // per class: exclusive prefix over warps
            int32_t run = s_carry[threadIdx.x];
            for (int w = 0; w < kW; ++w) {
                const int32_t v = s_wc[w][threadIdx.x];
                s_wc[w][threadIdx.x] = run;
                run += v;
            }
            s_carry[threadIdx.x] = run;
        }
        __syncthreads();
        if (c >= 0) pos[i] = s_wc[warp][c] + __popc(mine & ((1u << lane) - 1u));
        __syncthreads();                                  // s_wc is rewritten by the next chunk
    }
}

// The record of token block blk, written at its launch position pos[blk].
__global__ void __launch_bounds__(kTokThreads, kTokMinBlocks)
tdp_cond_record_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, const int32_t *__restrict__ slot,
                       const int32_t *__restrict__ pos, int32_t *__restrict__ recs)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    int32_t *rec = reinterpret_cast<int32_t *>(dsm + rows_layout(g.nt).rec);
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t blk = blockIdx.x;
    const int32_t nkb = (N + kTok - 1) / kTok;
    const int32_t b = blk / nkb, k0 = (blk - b * nkb) * kTok;
    const tok_rows tr = rows_from_slots(g, N, ncap, slot, blk, b, k0, dsm, rec);
    int32_t *dst = recs + (int64_t)pos[blk] * rec_ints(g.nt);
    for (int32_t i = threadIdx.x; i < kRecHead + tr.R; i += kTokThreads) dst[i] = rec[i];
}

// Block i = the token block whose record is the i-th (tdp_cond_rows.cuh's cond_record_block).
template <int BF16, int CR>
__global__ void __launch_bounds__(kTokThreads, kTokMinBlocks)
tdp_cond_blend_rec_kernel(int32_t nt, int32_t N, uint32_t nrows, int32_t CV, const int32_t *__restrict__ recs,
                          const uint4 *__restrict__ Ycond, uint4 *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    cond_record_block<BF16, CR>(nt, N, (int32_t)gridDim.x, nrows, CV, recs, Ycond, out, blockIdx.x, dsm);
}

// Token blocks of a problem and its record layout; TDP_OK when the records apply.
tdp_status rec_shape(const tdp_geom &g, int32_t N, int64_t *blocks)
{
    if (N < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "N must be >= 0");
    if (g.nt > kStageTiles) return tdp_fail(TDP_ERR_TOO_LARGE, "conditioning records take at most 256 tiles");
    *blocks = (int64_t)g.B * ((N + kTok - 1) / kTok);
    if (*blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "too many token blocks");
    return TDP_OK;
}

}  // namespace

extern "C" tdp_status tdp_cond_records_size(tdp_plan_t plan, int32_t N, int64_t *ints)
{
    if (!plan || !ints) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan or ints");
    int64_t G = 0;
    const tdp_status st = rec_shape(plan->g, N, &G);
    if (st != TDP_OK) return st;
    *ints = G * rec_ints(plan->g.nt) + G;
    return tdp_ok();
}

extern "C" tdp_status tdp_cond_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *slot, int32_t *recs,
                                       tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need ncap >= 1");
    int64_t G = 0;
    const tdp_status st = rec_shape(g, N, &G);
    if (st != TDP_OK) return st;
    if (G == 0) return tdp_ok();
    if (!slot || !recs) return tdp_fail(TDP_ERR_INVALID_ARG, "null slot or recs");
    if (!tdp_aligned(slot, 4) || !tdp_aligned(recs, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "slot needs 4-byte, recs 16-byte alignment");
    if ((uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap > 0xffffffffull)
        return tdp_fail(TDP_ERR_TOO_LARGE, "rows of Ycond numbered past 2^32");
    int32_t *pos = recs + G * rec_ints(g.nt);
    const size_t smem = rows_layout(g.nt).bytes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = tdp_launch_smem(true, tdp_cond_count_kernel, (unsigned)G, kTokThreads, smem, s, g, N, ncap,
                                      slot, pos);
    if (err == cudaSuccess) err = tdp_launch(true, tdp_cond_order_kernel, 1, kOrderThreads, s, (int32_t)G, pos);
    if (err == cudaSuccess)
        err = tdp_launch_smem(true, tdp_cond_record_kernel, (unsigned)G, kTokThreads, smem, s, g, N, ncap, slot,
                              static_cast<const int32_t *>(pos), recs);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_cond_blend_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *recs,
                                             const void *Ycond, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need ncap >= 1");
    int64_t G = 0;
    const tdp_status st = rec_shape(g, N, &G);
    if (st != TDP_OK) return st;
    if (G == 0) return tdp_ok();
    const uint64_t nrows = (uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap;
    if (nrows > 0xffffffffull) return tdp_fail(TDP_ERR_TOO_LARGE, "rows of Ycond numbered past 2^32");
    if (!recs || !Ycond || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null recs, Ycond or out");
    if (!tdp_aligned(recs, 16) || !tdp_aligned(Ycond, 16) || !tdp_aligned(out, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "recs, Ycond and out need 16-byte alignment");
    const int32_t CV = (g.C * g.esize) >> 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    cudaError_t err;
    if (g.nt >= kRecRowsTiles) {
        const size_t smem = rows_layout(g.nt, kRecRows).bytes;
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_cond_blend_rec_kernel<1, kRecRows>, (unsigned)G, kTokThreads, smem, s,
                                    g.nt, N, (uint32_t)nrows, CV, recs, y, o)
                  : tdp_launch_smem(true, tdp_cond_blend_rec_kernel<0, kRecRows>, (unsigned)G, kTokThreads, smem, s,
                                    g.nt, N, (uint32_t)nrows, CV, recs, y, o);
    } else {
        const size_t smem = rows_layout(g.nt).bytes;
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_cond_blend_rec_kernel<1, kChunkRows>, (unsigned)G, kTokThreads, smem, s,
                                    g.nt, N, (uint32_t)nrows, CV, recs, y, o)
                  : tdp_launch_smem(true, tdp_cond_blend_rec_kernel<0, kChunkRows>, (unsigned)G, kTokThreads, smem, s,
                                    g.nt, N, (uint32_t)nrows, CV, recs, y, o);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
