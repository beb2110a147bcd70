// tdp_blend.cu -- the blend entry points: tdp_blend (the gather pass of
// tdp_blend_row.cuh, a block per latent row), and for round-robin ranks
// tdp_blend_partial and tdp_blend_store ("Tiled Data Parallelism (TDP)", section
// "What it is": overlaps are blended with trapezoidal masks summing to one and the
// blended tiles are summed into the final result).
#include <atomic>

#include "tdp.h"
#include "tdp_blend_row.cuh"
#include "tdp_internal.h"

namespace {

using namespace tdp_bl;
constexpr int kBlendMinBlocks = 6;   // blocks per SM the register budget is sized for

template <int BF16>
__global__ void __launch_bounds__(kBlendThreads, kBlendMinBlocks)
tdp_blend_kernel(const __grid_constant__ tdp_geom g, int32_t cv_shift, const uint4 *__restrict__ Yout,
                 uint4 *__restrict__ Z)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    blend_row<BF16>(g, cv_shift, Yout, Z, blockIdx.x, dsm);
}

// ---------------------------------------------------------------------------
// Partial blend for round-robin ranks ("What it is": tiles go to ranks round-robin and
// one all_reduce sums the ranks' blended tiles).  Block = one latent row (b, f, h); a
// thread takes one 16-byte input vector of a cell at a time, loads the covering tiles
// that rank `rank` owns (t % world == rank; at most 8, all loads in flight before the
// arithmetic) and writes their mask-weighted sum in fp32, in ascending t with the same
// operations as tdp_blend_kernel, or +0 where the rank owns no covering tile.  With
// world == 1 the sums are tdp_blend_kernel's before its final rounding.
// ---------------------------------------------------------------------------
constexpr int kPartialThreads = 128;

template <int BF16>
__global__ void __launch_bounds__(kPartialThreads)
tdp_blend_partial_kernel(const __grid_constant__ tdp_geom g, int32_t rank, int32_t world,
                         const uint4 *__restrict__ Yout, float4 *__restrict__ Zp)
{
    using VM = vec_math<BF16>;
    constexpr int kE = VM::kElems;                    // elements per 16-byte input vector
    __shared__ int64_t s_tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    __shared__ int32_t s_loW[TDP_MAX_TILES_PER_DIM], s_hiW[TDP_MAX_TILES_PER_DIM];
    tdp_pdl_trigger();
    for (int32_t i = threadIdx.x; i < g.d[2].n; i += blockDim.x) {
        s_loW[i] = g.d[2].lo[i];
        s_hiW[i] = g.d[2].hi[i];
    }
    const int32_t row = blockIdx.x;
    const int32_t h = row % g.H, f = (row / g.H) % g.F, b = row / (g.H * g.F);
    const tdp_row_combos rc = tdp_make_combos(g, f, h);
    tdp_fill_row_table(g, rc, b, f, h, s_tok, nullptr, nullptr, nullptr);   // ends with a barrier
    const int32_t nW = g.d[2].n, nH = g.d[1].n, oW = g.d[2].o;
    const int32_t CV = (g.C * g.esize) >> 4;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    tdp_pdl_wait();
    const int64_t zrow = ((int64_t)b * T + ((int64_t)f * g.H + h) * g.W) * CV;   // first input vector of the row
    const int32_t nvec = g.W * CV;
    for (int32_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int32_t w = v / CV, cv = v - w * CV;
        const tdp_cover cW = tdp_cover_tab(s_loW, s_hiW, nW, g.W, oW, w);
        const float r0 = tdp_weight(cW.num0, oW), r1 = tdp_weight(cW.num1, oW);
        uint4 y[TDP_MAX_COMBOS][2];
        bool own[TDP_MAX_COMBOS][2];
#pragma unroll
        for (int c = 0; c < TDP_MAX_COMBOS; ++c)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int32_t iW = k ? cW.i1 : cW.i0;
                const int32_t t = c < rc.nc && iW >= 0 ? (rc.iF(c) * nH + rc.iH(c)) * nW + iW : -1;
                own[c][k] = t >= 0 && t % world == rank;
                if (own[c][k]) y[c][k] = __ldcs(Yout + (s_tok[c * nW + iW] + w) * CV + cv);
            }
        float acc[kE];
#pragma unroll
        for (int e = 0; e < kE; ++e) acc[e] = 0.0f;
        bool first = true;
#pragma unroll
        for (int c = 0; c < TDP_MAX_COMBOS; ++c)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (!own[c][k]) continue;
                const float m = rc.rFH(c) * (k ? r1 : r0);
                if (first) VM::mul(acc, m, y[c][k]);           // the first term keeps the sign of zero
                else VM::fma(acc, m, y[c][k]);
                first = false;
            }
        float4 *dst = Zp + (zrow + v) * (kE / 4);
#pragma unroll
        for (int q = 0; q < kE / 4; ++q)
            __stcs(dst + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
    }
}

// Z[i] = Zsum[i] in the plan's dtype (round to nearest even for bf16): 8 (bf16) or 4 (fp32)
// elements per thread and step, grid-stride.
template <int BF16>
__global__ void __launch_bounds__(256)
tdp_blend_store_kernel(int64_t nvec, const float4 *__restrict__ Zsum, uint4 *__restrict__ Z)
{
    using VM = vec_math<BF16>;
    constexpr int kE = VM::kElems;
    tdp_pdl_trigger();
    tdp_pdl_wait();
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
        float a[kE];
#pragma unroll
        for (int q = 0; q < kE / 4; ++q) {
            const float4 x = __ldcs(Zsum + v * (kE / 4) + q);
            a[4 * q] = x.x;
            a[4 * q + 1] = x.y;
            a[4 * q + 2] = x.z;
            a[4 * q + 3] = x.w;
        }
        __stcs(Z + v, VM::pack(a));
    }
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per device (calls after the
// first with a given size make no attribute change).
template <typename K>
cudaError_t allow_blend_smem(K kernel, size_t bytes)
{
    static std::atomic<int> raised[2][64];
    const int which = kernel == reinterpret_cast<K>(tdp_blend_kernel<1>) ? 1 : 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && raised[which][dev].load(std::memory_order_relaxed) >= (int)bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess && dev < 64) {
        int cur = raised[which][dev].load(std::memory_order_relaxed);
        while (cur < (int)bytes && !raised[which][dev].compare_exchange_weak(cur, (int)bytes)) {
        }
    }
    return err;
}

}  // namespace

extern "C" tdp_status tdp_blend_partial(tdp_plan_t plan, int32_t rank, int32_t world, const void *Yout, float *Zp,
                                        tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (world < 1 || rank < 0 || rank >= world) return tdp_fail(TDP_ERR_INVALID_ARG, "need 0 <= rank < world");
    if (g.B == 0) return tdp_ok();
    if (!Yout || !Zp) return tdp_fail(TDP_ERR_INVALID_ARG, "null Yout or Zp");
    if (!tdp_aligned(Yout, 16) || !tdp_aligned(Zp, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "Yout and Zp must be 16-byte aligned");
    const unsigned rows = (unsigned)((int64_t)g.B * g.F * g.H);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Yout);
    float4 *z = reinterpret_cast<float4 *>(Zp);
    cudaError_t err = g.dtype == TDP_BF16
                          ? tdp_launch(true, tdp_blend_partial_kernel<1>, rows, kPartialThreads, s, g, rank, world, y, z)
                          : tdp_launch(true, tdp_blend_partial_kernel<0>, rows, kPartialThreads, s, g, rank, world, y, z);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_blend_store(tdp_plan_t plan, int64_t n, const float *Zsum, void *Z, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    const int64_t per = 16 / g.esize;                 // elements per 16-byte output vector
    if (n < 0 || n % per != 0) return tdp_fail(TDP_ERR_INVALID_ARG, "n must be >= 0 and a multiple of 16 bytes of Z");
    if (n == 0) return tdp_ok();
    if (!Zsum || !Z) return tdp_fail(TDP_ERR_INVALID_ARG, "null Zsum or Z");
    if (!tdp_aligned(Zsum, 16) || !tdp_aligned(Z, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "Zsum and Z must be 16-byte aligned");
    const int64_t nvec = n / per;
    int64_t blocks = (nvec + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float4 *a = reinterpret_cast<const float4 *>(Zsum);
    uint4 *z = reinterpret_cast<uint4 *>(Z);
    cudaError_t err = g.dtype == TDP_BF16 ? tdp_launch(true, tdp_blend_store_kernel<1>, (unsigned)blocks, 256, s, nvec, a, z)
                                          : tdp_launch(true, tdp_blend_store_kernel<0>, (unsigned)blocks, 256, s, nvec, a, z);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_blend(tdp_plan_t plan, const void *Yout, void *Z, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (g.B == 0) return tdp_ok();
    if (!Yout || !Z) return tdp_fail(TDP_ERR_INVALID_ARG, "null Yout or Z");
    if (!tdp_aligned(Yout, 16) || !tdp_aligned(Z, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "Yout and Z must be 16-byte aligned");
    const int32_t CV = (g.C * g.esize) >> 4;
    const int32_t cv_shift = (CV & (CV - 1)) == 0 ? __builtin_ctz((unsigned)CV) : -1;
    const unsigned rows = (unsigned)((int64_t)g.B * g.F * g.H);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Yout);
    uint4 *z = reinterpret_cast<uint4 *>(Z);
    // the W-cell table is sized to the row (up to kWTab cells), so that short rows leave
    // room for more blocks per SM
    const size_t wsmem = blend_smem(g);
    cudaError_t err = g.dtype == TDP_BF16 ? allow_blend_smem(tdp_blend_kernel<1>, wsmem) : allow_blend_smem(tdp_blend_kernel<0>, wsmem);
    if (err == cudaSuccess)
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_blend_kernel<1>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z)
                  : tdp_launch_smem(true, tdp_blend_kernel<0>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
