// tdp_post.cu -- the post-model stage in one call: the blend of the tile outputs into
// the latent and the conditioning-token output reduction ("Tiled Data Parallelism
// (TDP)", section "What it is": the blended tiles are summed into the final result;
// "Shared negative (reference) positions": a conditioning token's outputs weigh
// 1/(number of tiles that kept it)).
//
// tdp_blend_cond_kernel is one grid of two kinds of block, both 128 threads: latent rows
// (tdp_blend_row.cuh's blend_row) and conditioning-token blocks (tdp_cond_rows.cuh's
// cond_rows_block).  The token blocks are latency-bound and the rows bandwidth-bound, so
// the token blocks sit behind two device-fulls of rows in block order: they start once
// the rows stream at full rate and run beside them instead of after them.  Every output
// is bit for bit what tdp_blend and tdp_cond_blend write.
#include <algorithm>
#include <atomic>

#include "tdp.h"
#include "tdp_blend_row.cuh"
#include "tdp_cond_rows.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kPostThreads = 128;
constexpr int kPostMinBlocks = 6;
static_assert(tdp_bl::kBlendThreads == kPostThreads && tdp_cr::kTokThreads == kPostThreads,
              "rows and token blocks share one launch");

// Blocks [0, fpos): rows 0..fpos-1; [fpos, fpos + ncond): conditioning-token blocks;
// the rest: rows fpos.. .
template <int BF16>
__global__ void __launch_bounds__(kPostThreads, kPostMinBlocks)
tdp_blend_cond_kernel(const __grid_constant__ tdp_geom g, int32_t cv_shift, const uint4 *__restrict__ Yout,
                      uint4 *__restrict__ Z, int32_t N, int32_t ncap, int32_t CV,
                      const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot, uint4 *__restrict__ outc,
                      int32_t fpos, int32_t ncond)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    const int32_t blk = blockIdx.x;
    if (blk >= fpos && blk < fpos + ncond) {
        tdp_cr::cond_rows_block<BF16>(g, N, ncap, CV, Ycond, slot, outc, blk - fpos, dsm);
        return;
    }
    tdp_bl::blend_row<BF16>(g, cv_shift, Yout, Z, blk < fpos ? blk : blk - ncond, dsm);
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per device (calls after the
// first with a given size make no attribute change), and return the blocks of it that
// fit on the whole device at that size (0 on error).
template <typename K>
int64_t prepare_post(K kernel, int which, size_t bytes, cudaError_t *err)
{
    static std::atomic<int> raised[2][64];
    int dev = 0, sms = 0, per_sm = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    if (dev >= 64 || raised[which][dev].load(std::memory_order_relaxed) < (int)bytes) {
        *err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (*err != cudaSuccess) return 0;
        if (dev < 64) {
            int cur = raised[which][dev].load(std::memory_order_relaxed);
            while (cur < (int)bytes && !raised[which][dev].compare_exchange_weak(cur, (int)bytes)) {
            }
        }
    }
    *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (*err == cudaSuccess) *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kPostThreads, bytes);
    return *err == cudaSuccess ? (int64_t)per_sm * sms : 0;
}

}  // namespace

extern "C" tdp_status tdp_blend_cond(tdp_plan_t plan, const void *Yout, void *Z, int32_t N, int32_t ncap,
                                     const void *Ycond, const int32_t *slot, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (N < 0 || ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need N >= 0 and ncap >= 1");
    if (g.B == 0) return tdp_ok();
    if (!Yout || !Z) return tdp_fail(TDP_ERR_INVALID_ARG, "null Yout or Z");
    if (!tdp_aligned(Yout, 16) || !tdp_aligned(Z, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "Yout and Z must be 16-byte aligned");
    if (N == 0) return tdp_blend(plan, Yout, Z, stream);
    if (!Ycond || !slot || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null Ycond, slot or out");
    if (!tdp_aligned(Ycond, 16) || !tdp_aligned(out, 16) || !tdp_aligned(slot, 4))
        return tdp_fail(TDP_ERR_MISALIGNED, "Ycond and out need 16-byte, slot 4-byte alignment");
    if (g.nt > tdp_cr::kStageTiles || (uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap > 0xffffffffull) {
        // beyond the token-block routine's range: the two calls one after the other
        const tdp_status st = tdp_blend(plan, Yout, Z, stream);
        return st != TDP_OK ? st : tdp_cond_blend(plan, N, ncap, Ycond, slot, out, stream);
    }
    const int64_t rows = (int64_t)g.B * g.F * g.H;
    const int64_t ncond = (int64_t)g.B * ((N + tdp_cr::kTok - 1) / tdp_cr::kTok);
    if (rows + ncond > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "post-model grid too large");
    const int32_t CV = (g.C * g.esize) >> 4;
    const int32_t cv_shift = (CV & (CV - 1)) == 0 ? __builtin_ctz((unsigned)CV) : -1;
    const size_t smem = std::max(tdp_bl::blend_smem(g), tdp_cr::rows_layout(g.nt).bytes);
    cudaError_t err = cudaSuccess;
    const int64_t resident = g.dtype == TDP_BF16 ? prepare_post(tdp_blend_cond_kernel<1>, 1, smem, &err)
                                                 : prepare_post(tdp_blend_cond_kernel<0>, 0, smem, &err);
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    // token blocks go behind two device-fulls of rows
    const int64_t fpos = std::min<int64_t>(rows, 2 * resident);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const unsigned grid = (unsigned)(rows + ncond);
    const uint4 *y = reinterpret_cast<const uint4 *>(Yout);
    uint4 *z = reinterpret_cast<uint4 *>(Z);
    const uint4 *yc = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    err = g.dtype == TDP_BF16
              ? tdp_launch_smem(true, tdp_blend_cond_kernel<1>, grid, kPostThreads, smem, s, g, cv_shift, y, z, N, ncap,
                                CV, yc, slot, o, (int32_t)fpos, (int32_t)ncond)
              : tdp_launch_smem(true, tdp_blend_cond_kernel<0>, grid, kPostThreads, smem, s, g, cv_shift, y, z, N, ncap,
                                CV, yc, slot, o, (int32_t)fpos, (int32_t)ncond);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
