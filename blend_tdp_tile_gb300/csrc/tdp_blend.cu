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
// one all_reduce sums the ranks' blended tiles).  Block = one latent row (b, f, h), the
// blend's row routine in its partial mode: the loads of the covering tiles rank `rank`
// owns (t % world == rank) go through the same shared-memory slots, and each output is
// their mask-weighted sum in fp32, in ascending t with tdp_blend_kernel's operations, or
// +0 where the rank owns no covering tile.  With world == 1 the sums are tdp_blend_kernel's
// before its final rounding.
// ---------------------------------------------------------------------------
template <int BF16>
__global__ void __launch_bounds__(kBlendThreads, kBlendMinBlocks)
tdp_blend_partial_kernel(const __grid_constant__ tdp_geom g, int32_t cv_shift, int32_t rank, int32_t world,
                         const uint4 *__restrict__ Yout, float4 *__restrict__ Zp)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    blend_row<BF16, 1>(g, cv_shift, Yout, Zp, blockIdx.x, dsm, rank, world);
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
// first with a given size make no attribute change); `which` names the kernel (0, 1: the
// blend in f32, bf16; 2, 3: the partial blend).
template <typename K>
cudaError_t allow_blend_smem(K kernel, int which, size_t bytes)
{
    static std::atomic<int> raised[4][64];
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
    const int32_t CV = (g.C * g.esize) >> 4;
    const int32_t cv_shift = (CV & (CV - 1)) == 0 ? __builtin_ctz((unsigned)CV) : -1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Yout);
    float4 *z = reinterpret_cast<float4 *>(Zp);
    const size_t wsmem = blend_smem(g);
    cudaError_t err = g.dtype == TDP_BF16 ? allow_blend_smem(tdp_blend_partial_kernel<1>, 3, wsmem)
                                          : allow_blend_smem(tdp_blend_partial_kernel<0>, 2, wsmem);
    if (err == cudaSuccess)
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_blend_partial_kernel<1>, rows, kBlendThreads, wsmem, s, g, cv_shift, rank,
                                    world, y, z)
                  : tdp_launch_smem(true, tdp_blend_partial_kernel<0>, rows, kBlendThreads, wsmem, s, g, cv_shift, rank,
                                    world, y, z);
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
    cudaError_t err = g.dtype == TDP_BF16 ? allow_blend_smem(tdp_blend_kernel<1>, 1, wsmem)
                                          : allow_blend_smem(tdp_blend_kernel<0>, 0, wsmem);
    if (err == cudaSuccess)
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_blend_kernel<1>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z)
                  : tdp_launch_smem(true, tdp_blend_kernel<0>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
