// tdp_blend.cu -- mask-weighted accumulation of all tile outputs into the
// full latent ("Tiled Data Parallelism (TDP)", section "What it is": overlaps
// are blended with trapezoidal masks summing to one and the blended tiles are
// summed into the final result; the page's cross-rank all_reduce becomes,
// with every tile on this GPU, one gather pass).
//
// Gather form.  A block owns one latent row (b, f, h).  Once per row it builds
// in shared memory the token offsets of the row inside every covering tile
// (at most 2 F-tiles x 2 H-tiles = 4 "combos", times the W-tiles) and a table
// of the (at most 2) W-tiles covering each cell with their ramp weights, so
// the per-vector work is table lookups, at most 8 independent 16-byte loads
// issued back to back, fp32 FMAs in ascending tile order and one streaming
// store.  Every tile-output byte is read exactly once and every latent byte
// written once: no atomics, no scratch memory, no inter-block waits.  The
// loads in flight bound a register-staged gather, so on rows with at most two
// F/H combos a thread takes four (one combo) or two (two combos) vectors per
// pass, up to 8 loads in flight, with 80 registers and 24 warps per SM (six
// 128-thread blocks, so that more rows are in flight at once).
#include <atomic>

#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kBlendThreads = 128;
constexpr int kWTab = 1024;      // cells of the per-row W table built per pass
constexpr int kBlendMinBlocks = 6;   // blocks per SM the register budget is sized for
constexpr size_t kBlendStage = 2 * 8 * kBlendThreads * 16;   // two passes of eight 16-byte slots per thread

// W-coverage of one cell: tiles iW0 (low 16 bits) and iW1 + 1 (high 16 bits,
// 0 = none) and their ramp weights.
struct __align__(16) tdp_wcell {
    int32_t iw;
    float r0, r1;
    int32_t pad;
};

template <int BF16>
struct vec_math;

template <>
struct vec_math<0> {     // 4 x fp32
    static constexpr int kElems = 4;
    __device__ static void mul(float (&a)[4], float m, const uint4 &y)
    {
        a[0] = m * __uint_as_float(y.x);
        a[1] = m * __uint_as_float(y.y);
        a[2] = m * __uint_as_float(y.z);
        a[3] = m * __uint_as_float(y.w);
    }
    __device__ static void fma(float (&a)[4], float m, const uint4 &y)
    {
        a[0] = fmaf(m, __uint_as_float(y.x), a[0]);
        a[1] = fmaf(m, __uint_as_float(y.y), a[1]);
        a[2] = fmaf(m, __uint_as_float(y.z), a[2]);
        a[3] = fmaf(m, __uint_as_float(y.w), a[3]);
    }
    __device__ static uint4 pack(const float (&a)[4])
    {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

template <>
struct vec_math<1> {     // 8 x bf16
    static constexpr int kElems = 8;
    __device__ static void mul(float (&a)[8], float m, const uint4 &y)
    {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = m * tdp_bf16_lo(w[i]);
            a[2 * i + 1] = m * tdp_bf16_hi(w[i]);
        }
    }
    __device__ static void fma(float (&a)[8], float m, const uint4 &y)
    {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = fmaf(m, tdp_bf16_lo(w[i]), a[2 * i]);
            a[2 * i + 1] = fmaf(m, tdp_bf16_hi(w[i]), a[2 * i + 1]);
        }
    }
    __device__ static uint4 pack(const float (&a)[8])
    {
        return make_uint4(tdp_pack_bf16x2(a[0], a[1]), tdp_pack_bf16x2(a[2], a[3]),
                          tdp_pack_bf16x2(a[4], a[5]), tdp_pack_bf16x2(a[6], a[7]));
    }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int BF16>
__global__ void __launch_bounds__(kBlendThreads, kBlendMinBlocks)
tdp_blend_kernel(const __grid_constant__ tdp_geom g, int32_t cv_shift, const uint4 *__restrict__ Yout,
                 uint4 *__restrict__ Z)
{
    using VM = vec_math<BF16>;
    __shared__ int64_t s_tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
    extern __shared__ __align__(16) unsigned char dsm[];
    // dynamic: the W-cell table (min(W, kWTab) cells), then the load slots of the passes
    tdp_wcell *s_w = reinterpret_cast<tdp_wcell *>(dsm);
    const int32_t wtab = g.W < kWTab ? g.W : kWTab;
    unsigned char *dsm_stage = dsm + (size_t)wtab * sizeof(tdp_wcell);
    const uint32_t stage = static_cast<uint32_t>(__cvta_generic_to_shared(dsm_stage));
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

    const int32_t nW = g.d[2].n, oW = g.d[2].o;
    const int32_t CV = (g.C * g.esize) >> 4;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    // tile-row offsets in 16-byte vectors: cell w, vector cv of (combo c, W-tile iW)
    // sits at Yout + s_tok[c * nW + iW] + w * CV + cv
    for (int32_t e = threadIdx.x; e < rc.nc * nW; e += blockDim.x) s_tok[e] *= CV;
    const int32_t nc = rc.nc;
    float rFH[TDP_MAX_COMBOS];
#pragma unroll
    for (int c = 0; c < TDP_MAX_COMBOS; ++c) rFH[c] = c < nc ? rc.rFH(c) : 0.0f;

    tdp_pdl_wait();                                   // Yout written by the work before

    for (int32_t wbase = 0; wbase < g.W; wbase += kWTab) {
        const int32_t wn = min(kWTab, g.W - wbase);
        for (int32_t i = threadIdx.x; i < wn; i += blockDim.x) {
            const tdp_cover cW = tdp_cover_tab(s_loW, s_hiW, nW, g.W, oW, wbase + i);
            tdp_wcell e;
            e.iw = cW.i0 | ((cW.i1 + 1) << 16);
            e.r0 = tdp_weight(cW.num0, oW);
            e.r1 = tdp_weight(cW.num1, oW);
            e.pad = 0;
            s_w[i] = e;
        }
        __syncthreads();
        // vector v of this pass is cell wbase + v / CV: at ybase + tile offset + v
        const uint4 *ybase = Yout + (int64_t)wbase * CV;
        uint4 *zbase = Z + ((int64_t)b * T + ((int64_t)f * g.H + h) * g.W + wbase) * CV;
        const int32_t nvec = wn * CV;
        // Eight load slots per pass, copied global -> shared memory with cp.async (no
        // registers held while in flight), two passes' slots per thread: a thread issues
        // pass p + 1's copies before it sums pass p.  Slot s of a pass is W-tile s & 1 of
        // combo (s >> 1) & (nc - 1) of the pass's vector s >> (1 + log2 nc): 4, 2 or 1
        // vectors per pass for 1, 2 or 4 combos.  Each sum is formed in ascending tile
        // order, combo by combo, as in tdp_blend's definition.
        const int32_t lq = 1 + (nc >> 1);                 // log2 of the slots per vector
        const int32_t step = (8 >> lq) * (int32_t)blockDim.x;
        auto issue = [&](int32_t v0, int32_t buf) {
#pragma unroll
            for (int sl = 0; sl < 8; ++sl) {
                const int32_t v = v0 + (sl >> lq) * (int32_t)blockDim.x;
                if (v < nvec) {
                    const int32_t iw = s_w[cv_shift >= 0 ? (v >> cv_shift) : v / CV].iw;
                    const int32_t iWx = (sl & 1) ? (iw >> 16) - 1 : (iw & 0xffff);
                    if (iWx >= 0)
                        cp_async16(stage + ((buf * 8 + sl) * kBlendThreads + threadIdx.x) * 16u,
                                   ybase + s_tok[((sl >> 1) & (nc - 1)) * nW + iWx] + v);
                }
            }
            cp_async_commit();
        };
        int32_t buf = 0;
        if ((int32_t)threadIdx.x < nvec) issue(threadIdx.x, 0);
        for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += step, buf ^= 1) {
            if (v0 + step < nvec) {
                issue(v0 + step, buf ^ 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            const uint4 *sb = reinterpret_cast<const uint4 *>(dsm_stage) + (buf * 8) * kBlendThreads + threadIdx.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t v = v0 + q * (int32_t)blockDim.x;
                if (q >= (8 >> lq) || v >= nvec) break;
                const tdp_wcell e = s_w[cv_shift >= 0 ? (v >> cv_shift) : v / CV];
                const bool two = (e.iw >> 16) != 0;
                const int32_t s0 = q << lq;
                float acc[VM::kElems];
                VM::mul(acc, rFH[0] * e.r0, sb[s0 * kBlendThreads]);          // the first term keeps the sign of zero
                if (two) VM::fma(acc, rFH[0] * e.r1, sb[(s0 + 1) * kBlendThreads]);
#pragma unroll
                for (int c = 1; c < TDP_MAX_COMBOS; ++c) {
                    if (c < nc) {
                        VM::fma(acc, rFH[c] * e.r0, sb[(s0 + 2 * c) * kBlendThreads]);
                        if (two) VM::fma(acc, rFH[c] * e.r1, sb[(s0 + 2 * c + 1) * kBlendThreads]);
                    }
                }
                __stcs(zbase + v, VM::pack(acc));
            }
        }
        __syncthreads();   // the table is rebuilt for the next cells
    }
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
    const size_t wsmem = (size_t)(g.W < kWTab ? g.W : kWTab) * sizeof(tdp_wcell) + kBlendStage;
    cudaError_t err = g.dtype == TDP_BF16 ? allow_blend_smem(tdp_blend_kernel<1>, wsmem) : allow_blend_smem(tdp_blend_kernel<0>, wsmem);
    if (err == cudaSuccess)
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_blend_kernel<1>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z)
                  : tdp_launch_smem(true, tdp_blend_kernel<0>, rows, kBlendThreads, wsmem, s, g, cv_shift, y, z);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
