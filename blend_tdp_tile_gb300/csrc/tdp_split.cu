// tdp_split.cu -- TDP tile split with tile positions and position
// normalisation ("Tiled Data Parallelism (TDP)", sections "What it is" and
// "Position normalization"), alone (tdp_split) or fused with the
// conditioning-token filter (tdp_split_filter, which also finds the bounds).
//
// The split is in scatter form: each latent row (b, f, h) is read ONCE with
// 16-byte loads and written to every tile row that holds it (at most
// 2 x 2 x 2 tiles); its positions likewise, shifted by the tiles' mn when
// normalising.  The scatter form reads the latent once instead of once per
// covering tile, so the split moves B*T*C + B*sum(T_t)*C elements, its
// algorithmic minimum.  The same split through the Tensor Memory Accelerator
// (bulk-tensor loads of tile-row segments into shared memory, bulk stores to the
// tiles) is tdp_split_tma in tdp_split_tma.cu: bit-identical, and on the large
// workload (64x128x192x128 bf16, 2x8x8 tiles) 0.32 ms against this kernel's 0.29 ms,
// its latent copy alone 0.260 ms against 0.267 ms.  These register-staged stores stay
// the default.
//
// tdp_split_filter runs the whole pre-model stage in three launches:
//   1. tdp_bounds_init_kernel   (plain launch)
//   2. tdp_bounds_kernel        (dependent launch; mn / mx)
//   3. tdp_split_filter_kernel  (dependent launch), one grid of three block kinds:
//        split rows     copy their latent row BEFORE waiting on the bounds kernel
//                       (the latent does not depend on it, and the kernels ahead of
//                       it in this call start only after all earlier work in the
//                       stream), then wait and write the normalised positions;
//        filter blocks  one per (tile, batch item): wait, then keep test, keep
//                       bytes and stable compaction of all N tokens;
//        count blocks   wait, then the per-token count of keeping tiles.
//      Filter and count blocks sit after the first split rows in block order, so
//      they start once the bounds are done and run beside the HBM-bound copy.
//      (Positions in blocks of their own, so that no split row waits, were slower:
//      each such block rebuilt its row tables for little work.)
#include <algorithm>
#include <atomic>

#include "tdp.h"
#include "tdp_filter.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitUnroll = 4;      // latent vectors each thread loads before storing any
static_assert(kSplitThreads == tdp_filt::kThreads, "split and filter blocks share one launch");

struct split_smem {
    int64_t tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    int64_t qpos[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    int64_t Tt[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    int32_t tb[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    int32_t loW[TDP_MAX_TILES_PER_DIM], hiW[TDP_MAX_TILES_PER_DIM];
};

// The row table of latent row `row` = (b, f, h) in shared memory, with the
// positions' part when `positions` is set.  Whole block; ends with a barrier.
struct split_row_id {
    int32_t b, f, h;
    tdp_row_combos rc;
};

__device__ __forceinline__ split_row_id split_table(const tdp_geom &g, int32_t row, bool positions, split_smem &sm)
{
    split_row_id r;
    r.h = row % g.H;
    r.f = (row / g.H) % g.F;
    r.b = row / (g.H * g.F);
    for (int32_t i = threadIdx.x; i < g.d[2].n; i += blockDim.x) {
        sm.loW[i] = g.d[2].lo[i];
        sm.hiW[i] = g.d[2].hi[i];
    }
    r.rc = tdp_make_combos(g, r.f, r.h);
    tdp_fill_row_table(g, r.rc, r.b, r.f, r.h, sm.tok, positions ? sm.qpos : nullptr, positions ? sm.Tt : nullptr,
                       positions ? sm.tb : nullptr);   // ends with a barrier
    return r;
}

// Latent of one row: every 16-byte vector is loaded once and stored to each tile
// holding it.  CV = 16-byte vectors per token.
__device__ __forceinline__ void split_latent(const tdp_geom &g, const split_row_id &r, const uint4 *__restrict__ X,
                                             uint4 *__restrict__ Y, const split_smem &sm)
{
    const int32_t nW = g.d[2].n, oW = g.d[2].o;
    const int32_t CV = (g.C * g.esize) >> 4;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    const int64_t gtok = (int64_t)r.b * T + ((int64_t)r.f * g.H + r.h) * g.W;   // token of (b,f,h,0)
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
            const tdp_cover cW = tdp_cover_tab(sm.loW, sm.hiW, nW, g.W, oW, w);
            for (int32_t c = 0; c < r.rc.nc; ++c) {
                __stcs(Y + (sm.tok[c * nW + cW.i0] + w) * CV + cv, xs[u]);
                if (cW.i1 >= 0) __stcs(Y + (sm.tok[c * nW + cW.i1] + w) * CV + cv, xs[u]);
            }
        }
    }
}

// Positions of one row: [B,3,T,2] -> tile-major [B,3,T_t,2], minus mn when normalising.
__device__ __forceinline__ void split_positions(const tdp_geom &g, const split_row_id &r,
                                                const int2 *__restrict__ P, int32_t normalize,
                                                int2 *__restrict__ Q, const int32_t *__restrict__ mn,
                                                const split_smem &sm)
{
    const int32_t nW = g.d[2].n, oW = g.d[2].o;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    for (int32_t q = threadIdx.x; q < 3 * g.W; q += blockDim.x) {
        const int32_t d = q / g.W, w = q - d * g.W;
        const int2 p = __ldcs(P + ((int64_t)r.b * 3 + d) * T + ((int64_t)r.f * g.H + r.h) * g.W + w);
        const tdp_cover cW = tdp_cover_tab(sm.loW, sm.hiW, nW, g.W, oW, w);
        for (int32_t c = 0; c < r.rc.nc; ++c) {
            for (int32_t k = 0; k < 2; ++k) {
                const int32_t iW = k ? cW.i1 : cW.i0;
                if (iW < 0) break;
                const int32_t e = c * nW + iW;
                int2 o = p;
                if (normalize) {
                    const int32_t m = __ldg(mn + (int64_t)sm.tb[e] * 3 + d);
                    o.x = (int32_t)((uint32_t)p.x - (uint32_t)m);
                    o.y = (int32_t)((uint32_t)p.y - (uint32_t)m);
                }
                Q[sm.qpos[e] + (int64_t)d * sm.Tt[e] + w] = o;   // default policy: neighbouring rows merge in L2
            }
        }
    }
}

// Block = one latent row (b, f, h): latent and positions.
__global__ void __launch_bounds__(kSplitThreads)
tdp_split_kernel(const __grid_constant__ tdp_geom g, const uint4 *__restrict__ X,
                 const int2 *__restrict__ P, int32_t normalize, uint4 *__restrict__ Y,
                 int2 *__restrict__ Q, const int32_t *__restrict__ mn)
{
    __shared__ split_smem sm;
    tdp_pdl_trigger();
    const split_row_id r = split_table(g, blockIdx.x, P != nullptr, sm);
    tdp_pdl_wait();
    split_latent(g, r, X, Y, sm);
    if (P) split_positions(g, r, P, normalize, Q, mn, sm);
}

// Blocks [0, fpos): split rows 0..fpos-1; [fpos, fpos + nfilt): filter blocks
// (tb = t*B + b); [fpos + nfilt, fpos + nfilt + ncount): count blocks; the rest:
// split rows fpos.. .  Split rows copy their latent before waiting on the bounds
// kernel (see the file header) and wait only for the normalised positions.
__global__ void __launch_bounds__(kSplitThreads, 4)
tdp_split_filter_kernel(const __grid_constant__ tdp_geom g, const uint4 *__restrict__ X,
                        const int2 *__restrict__ P, int32_t normalize, uint4 *__restrict__ Y,
                        int2 *__restrict__ Q, const int32_t *__restrict__ mn, const int32_t *__restrict__ mx,
                        const int2 *__restrict__ K, int32_t N, uint8_t *__restrict__ keep,
                        int32_t *__restrict__ idx, int32_t *__restrict__ count, int32_t *__restrict__ kcount,
                        int2 *__restrict__ Kout, int32_t *__restrict__ slot, int32_t fpos, int32_t nfilt,
                        int32_t ncount)
{
    __shared__ union {
        split_smem split;
        tdp_filt::compact_smem compact;
        tdp_filt::kcount_smem kc;
    } sm;
    tdp_pdl_trigger();
    const int32_t blk = blockIdx.x;
    if (blk >= fpos && blk < fpos + nfilt + ncount) {
        tdp_pdl_wait();                             // mn / mx final
        const int32_t r = blk - fpos;
        if (r < nfilt)
            tdp_filt::tb_block(g, K, N, mn, mx, normalize, r, keep, idx, count, Kout, slot, sm.compact);
        else
            tdp_filt::kcount_block(g, K, N, mn, mx, kcount, r - nfilt, sm.kc);
        return;
    }
    const split_row_id r = split_table(g, blk < fpos ? blk : blk - nfilt - ncount, true, sm.split);
    split_latent(g, r, X, Y, sm.split);
    tdp_pdl_wait();                                 // mn final from here on
    split_positions(g, r, P, normalize, Q, mn, sm.split);
}

// Split blocks resident on the whole device at once (cached per device).
int32_t resident_split_blocks()
{
    static std::atomic<int32_t> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int32_t v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tdp_split_filter_kernel, kSplitThreads, 0) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int32_t v = per_sm * sms;
    if (dev < 64 && v > 0) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

}  // namespace

tdp_status tdp_check_split_args(const tdp_geom &g, const void *X, const int32_t *P, const int32_t *mn,
                                int32_t normalize, const void *Y, const int32_t *Q)
{
    if ((P == nullptr) != (Q == nullptr)) return tdp_fail(TDP_ERR_INVALID_ARG, "P and Q must be both set or both NULL");
    if (P && normalize && !mn) return tdp_fail(TDP_ERR_INVALID_ARG, "normalising needs mn");
    if (g.B == 0) return TDP_OK;
    if (!X || !Y) return tdp_fail(TDP_ERR_INVALID_ARG, "null X or Y");
    if (!tdp_aligned(X, 16) || !tdp_aligned(Y, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "X and Y must be 16-byte aligned");
    if (P && (!tdp_aligned(P, 8) || !tdp_aligned(Q, 8) || !tdp_aligned(mn, 4)))
        return tdp_fail(TDP_ERR_MISALIGNED, "P, Q need 8-byte and mn 4-byte alignment");
    return TDP_OK;
}

extern "C" tdp_status tdp_split(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *mn,
                                int32_t normalize, void *Y, int32_t *Q, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    const tdp_status st = tdp_check_split_args(g, X, P, mn, normalize, Y, Q);
    if (st != TDP_OK) return st;
    if (g.B == 0) return tdp_ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    cudaError_t err = tdp_launch(true, tdp_split_kernel, (unsigned)rows, kSplitThreads, s, g,
                                 reinterpret_cast<const uint4 *>(X), reinterpret_cast<const int2 *>(P),
                                 P ? normalize : 0, reinterpret_cast<uint4 *>(Y), reinterpret_cast<int2 *>(Q), mn);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_split_filter(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *K,
                                       int32_t N, int32_t normalize, void *Y, int32_t *Q, int32_t *mn,
                                       int32_t *mx, uint8_t *keep, int32_t *idx, int32_t *count,
                                       int32_t *kcount, int32_t *Kout, int32_t *slot, tdp_stream_t stream)
{
    using namespace tdp_filt;
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (N < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "N must be >= 0");
    if (g.B == 0) return tdp_ok();
    if (!P || !Q) return tdp_fail(TDP_ERR_INVALID_ARG, "null P or Q");
    if (!mn || !mx) return tdp_fail(TDP_ERR_INVALID_ARG, "null mn or mx");
    const tdp_status st = tdp_check_split_args(g, X, P, mn, normalize, Y, Q);
    if (st != TDP_OK) return st;
    if (!count) return tdp_fail(TDP_ERR_INVALID_ARG, "null count");
    if (N > 0 && (!K || !keep || !idx || !kcount || !Kout))
        return tdp_fail(TDP_ERR_INVALID_ARG, "null K, keep, idx, kcount or Kout");
    if (!tdp_aligned(mx, 4) || !tdp_aligned(count, 4) ||
        (N > 0 && (!tdp_aligned(K, 8) || !tdp_aligned(Kout, 8) || !tdp_aligned(idx, 4) ||
                   !tdp_aligned(kcount, 4) || !tdp_aligned(slot, 4))))
        return tdp_fail(TDP_ERR_MISALIGNED, "K, Kout need 8-byte and int32 buffers 4-byte alignment");
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    const int64_t nfilt = (int64_t)g.nt * g.B;
    const int64_t ncount = (int64_t)g.B * ((N + kCountTok - 1) / kCountTok);
    if (rows + nfilt + ncount > 0x7fffffffLL || (int64_t)g.B * N * g.nt > ((int64_t)1 << 56))
        return tdp_fail(TDP_ERR_TOO_LARGE, "split / filter grid too large");
    // filter and count blocks go behind two device-fulls of split rows
    const int64_t fpos = std::min<int64_t>(rows, 2 * (int64_t)resident_split_blocks());
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = tdp_launch_bounds(g, P, mn, mx, s);
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_split_filter_kernel, (unsigned)(rows + nfilt + ncount), kSplitThreads, s, g,
                         reinterpret_cast<const uint4 *>(X), reinterpret_cast<const int2 *>(P), normalize,
                         reinterpret_cast<uint4 *>(Y), reinterpret_cast<int2 *>(Q),
                         static_cast<const int32_t *>(mn), static_cast<const int32_t *>(mx),
                         reinterpret_cast<const int2 *>(K), N, keep, idx, count, kcount,
                         reinterpret_cast<int2 *>(Kout), slot, (int32_t)fpos, (int32_t)nfilt, (int32_t)ncount);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
