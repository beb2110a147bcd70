// tdp_blend.cu -- mask-weighted accumulation of all tile outputs into the
// full latent ("Tiled Data Parallelism (TDP)", section "What it is": overlaps
// are blended with trapezoidal masks summing to one and the blended tiles are
// summed into the final result; the page's cross-rank all_reduce becomes,
// with every tile on this GPU, one gather pass).
//
// Gather form: a block owns one latent row (b, f, h); every 16-byte output
// vector reads its (at most 2 x 2 x 2) covering tile vectors, weights them with
// masks computed in registers from the ramp formula, accumulates in fp32 in
// ascending tile order and is stored once.  Each tile-output element is read
// exactly once over the whole launch, each latent element written once, no
// atomics and no scratch.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kBlendThreads = 256;
constexpr int kUnroll = 2;     // output vectors per thread in flight

template <int BF16>
struct vec_math;

template <>
struct vec_math<0> {           // 4 x fp32
    static constexpr int kElems = 4;
    __device__ static void fma(float (&acc)[4], float m, const uint4 &y)
    {
        acc[0] = fmaf(m, __uint_as_float(y.x), acc[0]);
        acc[1] = fmaf(m, __uint_as_float(y.y), acc[1]);
        acc[2] = fmaf(m, __uint_as_float(y.z), acc[2]);
        acc[3] = fmaf(m, __uint_as_float(y.w), acc[3]);
    }
    __device__ static void mul(float (&acc)[4], float m, const uint4 &y)
    {
        acc[0] = m * __uint_as_float(y.x);
        acc[1] = m * __uint_as_float(y.y);
        acc[2] = m * __uint_as_float(y.z);
        acc[3] = m * __uint_as_float(y.w);
    }
    __device__ static uint4 pack(const float (&a)[4])
    {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

template <>
struct vec_math<1> {           // 8 x bf16
    static constexpr int kElems = 8;
    __device__ static void fma(float (&acc)[8], float m, const uint4 &y)
    {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(m, tdp_bf16_lo(w[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(m, tdp_bf16_hi(w[i]), acc[2 * i + 1]);
        }
    }
    __device__ static void mul(float (&acc)[8], float m, const uint4 &y)
    {
        const uint32_t w[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = m * tdp_bf16_lo(w[i]);
            acc[2 * i + 1] = m * tdp_bf16_hi(w[i]);
        }
    }
    __device__ static uint4 pack(const float (&a)[8])
    {
        return make_uint4(tdp_pack_bf16x2(a[0], a[1]), tdp_pack_bf16x2(a[2], a[3]),
                          tdp_pack_bf16x2(a[4], a[5]), tdp_pack_bf16x2(a[6], a[7]));
    }
};

template <int BF16>
__global__ void __launch_bounds__(kBlendThreads)
tdp_blend_kernel(const __grid_constant__ tdp_geom g, const uint4 *__restrict__ Yout, uint4 *__restrict__ Z)
{
    using VM = vec_math<BF16>;
    __shared__ int64_t s_tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];

    const int32_t row = blockIdx.x;
    const int32_t h = row % g.H, f = (row / g.H) % g.F, b = row / (g.H * g.F);
    const tdp_row_combos rc = tdp_make_combos(g, f, h);
    tdp_fill_row_table(g, rc, b, f, h, s_tok, nullptr, nullptr, nullptr);

    const int32_t nW = g.d[2].n;
    const int32_t CV = (g.C * g.esize) >> 4;
    const int32_t nvec = g.W * CV;
    const int64_t T = (int64_t)g.F * g.H * g.W;
    uint4 *dst = Z + ((int64_t)b * T + ((int64_t)f * g.H + h) * g.W) * CV;

    for (int32_t v0 = threadIdx.x; v0 < nvec; v0 += kUnroll * blockDim.x) {
        // issue every load of kUnroll output vectors before any arithmetic
        uint4 y[kUnroll][2 * TDP_MAX_COMBOS];
        float m[kUnroll][2 * TDP_MAX_COMBOS];
        int32_t nterm[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t v = v0 + u * blockDim.x;
            nterm[u] = 0;
            if (v >= nvec) continue;
            const int32_t w = v / CV, cv = v - w * CV;
            const tdp_cover cW = tdp_cover_1d(g.d[2], w);
            const float rW0 = tdp_weight(cW.num0, g.d[2].o);
            const float rW1 = tdp_weight(cW.num1, g.d[2].o);
#pragma unroll
            for (int c = 0; c < TDP_MAX_COMBOS; ++c) {
                if (c < rc.nc) {
                    y[u][2 * c] = __ldcs(Yout + (s_tok[c * nW + cW.i0] + w) * CV + cv);
                    m[u][2 * c] = rc.rFH[c] * rW0;
                    if (cW.i1 >= 0) {
                        y[u][2 * c + 1] = __ldcs(Yout + (s_tok[c * nW + cW.i1] + w) * CV + cv);
                        m[u][2 * c + 1] = rc.rFH[c] * rW1;
                    }
                }
            }
            nterm[u] = cW.i1 >= 0 ? 2 : 1;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (nterm[u] == 0) continue;
            const int32_t v = v0 + u * blockDim.x;
            float acc[VM::kElems];
            VM::mul(acc, m[u][0], y[u][0]);                   // first term sets the sign of zero
#pragma unroll
            for (int c = 0; c < TDP_MAX_COMBOS; ++c) {
                if (c < rc.nc) {
                    if (c > 0) VM::fma(acc, m[u][2 * c], y[u][2 * c]);
                    if (nterm[u] == 2) VM::fma(acc, m[u][2 * c + 1], y[u][2 * c + 1]);
                }
            }
            __stcs(dst + v, VM::pack(acc));
        }
    }
}

}  // namespace

extern "C" tdp_status tdp_blend(tdp_plan_t plan, const void *Yout, void *Z, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (g.B == 0) return tdp_ok();
    if (!Yout || !Z) return tdp_fail(TDP_ERR_INVALID_ARG, "null Yout or Z");
    if (!tdp_aligned(Yout, 16) || !tdp_aligned(Z, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "Yout and Z must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const unsigned rows = (unsigned)((int64_t)g.B * g.F * g.H);
    if (g.dtype == TDP_BF16)
        tdp_blend_kernel<1><<<rows, kBlendThreads, 0, s>>>(g, reinterpret_cast<const uint4 *>(Yout),
                                                           reinterpret_cast<uint4 *>(Z));
    else
        tdp_blend_kernel<0><<<rows, kBlendThreads, 0, s>>>(g, reinterpret_cast<const uint4 *>(Yout),
                                                           reinterpret_cast<uint4 *>(Z));
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
