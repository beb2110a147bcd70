// tdp_cond.cu -- the two reductions over tiles besides the latent blend
// ("Tiled Data Parallelism (TDP)"):
//   tdp_cond_blend_kernel  each conditioning token's per-tile outputs averaged
//                          over the tiles that kept it ("Shared negative
//                          (reference) positions": weight 1/(tiles that kept it));
//   tdp_tile_mean_kernel   the audio latent averaged over all tiles ("What it
//                          is": audio is processed on every tile and averaged).
// Both are gather form and accumulate in fp32; no atomics, no scratch.  The
// conditioning blend adds each token's rows in ascending tile order (in runs of
// kListRows rows whose sums are added in order, for a token kept by many tiles);
// the tile mean adds the tiles of each quarter of the tile range in ascending
// order and then the four quarters' sums in order.
//
// tdp_cond_blend has two kernels.  With at most kStageTiles tiles (and rows of
// Ycond numbered below 2^32), a block takes kBlockTok consecutive tokens of one
// batch item: it stages their slots [tile][token] in shared memory (each tile's
// slots are one coalesced read) and lists per token, in ascending tile order,
// the rows of Ycond of the tiles that kept it.  A token kept by at most kLightRows tiles gets a group of lanes
// across its channel vectors that sums its rows one by one, kListRows loads
// in flight.  A token kept by more (a negative-time token is kept by every
// tile) gets the whole block: each group sums a run of kListRows consecutive
// rows of its list, and the runs' sums are added in order, so one such token
// does not hold its block for many rounds of loads.  With more than
// kStageTiles tiles, a warp per token reads the slots of 32 tiles at a time.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kMeanVecs = 64;     // output vectors per tile-mean block
constexpr int kMeanParts = 4;     // threads per output vector, each over a quarter of the tiles
constexpr int kMeanUnroll = 8;    // tile loads a tile-mean thread keeps in flight
constexpr int kStageTiles = 256;  // tiles the staged conditioning blend handles
constexpr int kBlockTok = 16;     // tokens per block of the staged conditioning blend
constexpr int kListRows = 8;      // row loads in flight per lane in the staged conditioning blend
constexpr int kLightRows = 16;    // kept tiles up to which a token is summed by one lane group

template <int BF16>
__device__ __forceinline__ void acc_add(float (&a)[8], const uint4 &y)
{
    const uint32_t w[4] = {y.x, y.y, y.z, y.w};
    if (BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] += tdp_bf16_lo(w[i]);
            a[2 * i + 1] += tdp_bf16_hi(w[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] += __uint_as_float(w[i]);
    }
}

template <int BF16>
__device__ __forceinline__ uint4 acc_div(const float (&a)[8], float n)
{
    if (BF16)
        return make_uint4(tdp_pack_bf16x2(__fdiv_rn(a[0], n), __fdiv_rn(a[1], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[2], n), __fdiv_rn(a[3], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[4], n), __fdiv_rn(a[5], n)),
                          tdp_pack_bf16x2(__fdiv_rn(a[6], n), __fdiv_rn(a[7], n)));
    return make_uint4(__float_as_uint(__fdiv_rn(a[0], n)), __float_as_uint(__fdiv_rn(a[1], n)),
                      __float_as_uint(__fdiv_rn(a[2], n)), __float_as_uint(__fdiv_rn(a[3], n)));
}

// Warp = one conditioning token (b, k).  Per round of 32 tiles, lane l loads the
// token's slot in tile t0 + l; a ballot gives the tiles that kept it, in
// ascending order, and their rows (lanes across the channel vectors) are loaded
// up to kRowsInFlight at a time and accumulated in that order.
constexpr int kRowsInFlight = 4;

template <int BF16>
__global__ void __launch_bounds__(kThreads)
tdp_cond_blend_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV,
                      const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot, uint4 *__restrict__ out)
{
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (tok >= (int64_t)g.B * N) return;                 // warp-uniform
    const int32_t b = (int32_t)(tok / N), k = (int32_t)(tok - (int64_t)b * N);
    for (int32_t cv0 = 0; cv0 < CV; cv0 += 32) {
        const int32_t cv = cv0 + lane;
        const bool act = cv < CV;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int32_t n = 0;
        for (int32_t t0 = 0; t0 < g.nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < g.nt ? __ldg(slot + ((int64_t)t * g.B + b) * N + k) : -1;
            uint32_t m = __ballot_sync(0xffffffffu, sl >= 0 && sl < ncap);
            while (m) {                                      // warp-uniform
                uint4 y[kRowsInFlight];
                int32_t got = 0;
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u) {
                    if (m) {
                        const int32_t j = __ffs(m) - 1;
                        m &= m - 1;
                        const int32_t sj = __shfl_sync(0xffffffffu, sl, j);
                        const int64_t tb = (int64_t)(t0 + j) * g.B + b;
                        if (act) y[u] = __ldcs(Ycond + (tb * ncap + sj) * CV + cv);
                        got = u + 1;
                    }
                }
#pragma unroll
                for (int u = 0; u < kRowsInFlight; ++u)
                    if (u < got && act) acc_add<BF16>(acc, y[u]);
                n += got;
            }
        }
        if (act) __stcs(out + tok * CV + cv, n > 0 ? acc_div<BF16>(acc, (float)n) : make_uint4(0u, 0u, 0u, 0u));
    }
}

struct cond_smem {
    int32_t slot[kStageTiles][kBlockTok + 1];      // +1: column reads spread over the banks
    uint32_t row[kBlockTok][kStageTiles];          // kept rows of Ycond per token, ascending tile
    int32_t len[kBlockTok];
    float part[8][kThreads];                       // run sums of a heavy token, one per lane
};

// Sum rows i0 .. i0 + kListRows - 1 (those below len) of token j's list into acc.
template <int BF16>
__device__ __forceinline__ void cond_rows(const cond_smem &sm, const uint4 *__restrict__ Ycond, int32_t CV,
                                          int32_t cv, int32_t j, int32_t i0, int32_t len, float (&acc)[8])
{
    uint4 y[kListRows];
#pragma unroll
    for (int u = 0; u < kListRows; ++u)
        if (i0 + u < len) y[u] = __ldcs(Ycond + (int64_t)sm.row[j][i0 + u] * CV + cv);
#pragma unroll
    for (int u = 0; u < kListRows; ++u)
        if (i0 + u < len) acc_add<BF16>(acc, y[u]);
}

// Block = tokens k0 .. k0 + kBlockTok - 1 of batch item b.
template <int BF16>
__global__ void __launch_bounds__(kThreads, 3)
tdp_cond_blend_staged_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV, int32_t lpt,
                             const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot,
                             uint4 *__restrict__ out)
{
    __shared__ cond_smem sm;
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t nkb = (N + kBlockTok - 1) / kBlockTok;
    const int32_t b = blockIdx.x / nkb, k0 = (blockIdx.x - b * nkb) * kBlockTok;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t nt = g.nt;
    // slots of the block's tokens in every tile, all of a thread's loads in flight
    // before any is stored
    {
        constexpr int kPer = kStageTiles * kBlockTok / kThreads;   // loads per thread
        constexpr int kStep = kThreads / kBlockTok;                 // tiles per pass of the block
        const int32_t j = threadIdx.x % kBlockTok;
        const bool tok_ok = k0 + j < N;
        const int32_t tb0 = threadIdx.x / kBlockTok;
        int32_t v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int32_t t = tb0 + u * kStep;
            v[u] = t < nt && tok_ok ? __ldg(slot + ((int64_t)t * g.B + b) * N + k0 + j) : -1;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int32_t t = tb0 + u * kStep;
            if (t < nt) sm.slot[t][j] = v[u];
        }
    }
    __syncthreads();
    // per token, the rows of the tiles that kept it, in ascending tile order
    for (int32_t j = warp; j < kBlockTok; j += kThreads / 32) {
        int32_t len = 0;
        for (int32_t t0 = 0; t0 < nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < nt ? sm.slot[t][j] : -1;
            const uint32_t m = __ballot_sync(0xffffffffu, sl >= 0 && sl < ncap);
            if ((m >> lane) & 1u)
                sm.row[j][len + __popc(m & ((1u << lane) - 1u))] = ((uint32_t)t * g.B + b) * (uint32_t)ncap + sl;
            len += __popc(m);
        }
        if (lane == 0) sm.len[j] = len;
    }
    __syncthreads();
    const int32_t groups = kThreads / lpt, grp = threadIdx.x / lpt, gl = threadIdx.x - grp * lpt;
    // light tokens: a group of lpt lanes per token, rows summed one by one in list order
    for (int32_t j = grp; j < kBlockTok && k0 + j < N; j += groups) {
        const int32_t len = sm.len[j];
        if (len > kLightRows) continue;
        const int64_t tok = (int64_t)b * N + k0 + j;
        for (int32_t cv = gl; cv < CV; cv += lpt) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int32_t i0 = 0; i0 < len; i0 += kListRows) cond_rows<BF16>(sm, Ycond, CV, cv, j, i0, len, acc);
            __stcs(out + tok * CV + cv, len > 0 ? acc_div<BF16>(acc, (float)len) : make_uint4(0u, 0u, 0u, 0u));
        }
    }
    // heavy tokens: the whole block; group q sums run q of kListRows consecutive rows,
    // group 0 adds the runs' sums in order
    for (int32_t j = 0; j < kBlockTok && k0 + j < N; ++j) {
        const int32_t len = sm.len[j];                // block-uniform
        if (len <= kLightRows) continue;
        const int64_t tok = (int64_t)b * N + k0 + j;
        for (int32_t cv0 = 0; cv0 < CV; cv0 += lpt) {
            const int32_t cv = cv0 + gl;
            const bool act = cv < CV;
            float tot[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int32_t r0 = 0; r0 < len; r0 += groups * kListRows) {
                float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (act) cond_rows<BF16>(sm, Ycond, CV, cv, j, r0 + grp * kListRows, len, part);
#pragma unroll
                for (int e = 0; e < 8; ++e) sm.part[e][threadIdx.x] = part[e];
                __syncthreads();
                if (grp == 0 && act) {
                    for (int32_t q = 0; q < groups && r0 + q * kListRows < len; ++q) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) tot[e] += sm.part[e][q * lpt + gl];
                    }
                }
                __syncthreads();
            }
            if (grp == 0 && act) __stcs(out + tok * CV + cv, acc_div<BF16>(tot, (float)len));
        }
    }
}

// Block = kMeanVecs output vectors of out[B, L]; thread (part p, vector v) sums
// tiles [p*nt/4, (p+1)*nt/4) in ascending order, kMeanUnroll loads in flight;
// part 0 adds the four sums in order and divides.
template <int BF16>
__global__ void __launch_bounds__(kMeanVecs * kMeanParts)
tdp_tile_mean_kernel(int32_t nt, int64_t nvec, const uint4 *__restrict__ A, uint4 *__restrict__ out)
{
    __shared__ float s_part[kMeanParts][8][kMeanVecs];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t vi = threadIdx.x % kMeanVecs, p = threadIdx.x / kMeanVecs;
    const int64_t v = (int64_t)blockIdx.x * kMeanVecs + vi;
    const int32_t ta = (int32_t)((int64_t)p * nt / kMeanParts), tz = (int32_t)((int64_t)(p + 1) * nt / kMeanParts);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (v < nvec) {
        for (int32_t t0 = ta; t0 < tz; t0 += kMeanUnroll) {
            uint4 y[kMeanUnroll];
#pragma unroll
            for (int u = 0; u < kMeanUnroll; ++u)
                if (t0 + u < tz) y[u] = __ldcs(A + (int64_t)(t0 + u) * nvec + v);
#pragma unroll
            for (int u = 0; u < kMeanUnroll; ++u)
                if (t0 + u < tz) acc_add<BF16>(acc, y[u]);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s_part[p][e][vi] = acc[e];
    __syncthreads();
    if (p == 0 && v < nvec) {
#pragma unroll
        for (int q = 1; q < kMeanParts; ++q)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += s_part[q][e][vi];
        __stcs(out + v, acc_div<BF16>(acc, (float)nt));
    }
}

}  // namespace

extern "C" tdp_status tdp_cond_blend(tdp_plan_t plan, int32_t N, int32_t ncap, const void *Ycond,
                                     const int32_t *slot, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (N < 0 || ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need N >= 0 and ncap >= 1");
    if (g.B == 0 || N == 0) return tdp_ok();
    if (!Ycond || !slot || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null Ycond, slot or out");
    if (!tdp_aligned(Ycond, 16) || !tdp_aligned(out, 16) || !tdp_aligned(slot, 4))
        return tdp_fail(TDP_ERR_MISALIGNED, "Ycond and out need 16-byte, slot 4-byte alignment");
    const int32_t CV = (g.C * g.esize) >> 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    cudaError_t err;
    if (g.nt <= kStageTiles && (uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap <= 0xffffffffull) {
        const int64_t blocks = (int64_t)g.B * ((N + kBlockTok - 1) / kBlockTok);
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
        int32_t lpt = 1;                                      // lanes per token: CV rounded up to 2^k, <= 32
        while (lpt < CV && lpt < 32) lpt *= 2;
        err = g.dtype == TDP_BF16
                  ? tdp_launch(true, tdp_cond_blend_staged_kernel<1>, (unsigned)blocks, kThreads, s, g, N, ncap, CV,
                               lpt, y, slot, o)
                  : tdp_launch(true, tdp_cond_blend_staged_kernel<0>, (unsigned)blocks, kThreads, s, g, N, ncap, CV,
                               lpt, y, slot, o);
    } else {
        const int64_t warps = (int64_t)g.B * N;              // one warp per conditioning token
        const int64_t blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
        err = g.dtype == TDP_BF16
                  ? tdp_launch(true, tdp_cond_blend_kernel<1>, (unsigned)blocks, kThreads, s, g, N, ncap, CV, y, slot, o)
                  : tdp_launch(true, tdp_cond_blend_kernel<0>, (unsigned)blocks, kThreads, s, g, N, ncap, CV, y, slot, o);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_tile_mean(tdp_plan_t plan, int64_t L, const void *A, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (L < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "L must be >= 0");
    if (g.B == 0 || L == 0) return tdp_ok();
    if (!A || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null A or out");
    if ((L * g.esize) % 16 != 0) return tdp_fail(TDP_ERR_MISALIGNED, "L * element size must be a multiple of 16");
    if (!tdp_aligned(A, 16) || !tdp_aligned(out, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "A and out must be 16-byte aligned");
    const int64_t nvec = (int64_t)g.B * L * g.esize / 16;
    const int64_t blocks = (nvec + kMeanVecs - 1) / kMeanVecs;
    if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "tile mean grid too large");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *a = reinterpret_cast<const uint4 *>(A);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    const unsigned threads = kMeanVecs * kMeanParts;
    cudaError_t err = g.dtype == TDP_BF16
                          ? tdp_launch(true, tdp_tile_mean_kernel<1>, (unsigned)blocks, threads, s, g.nt, nvec, a, o)
                          : tdp_launch(true, tdp_tile_mean_kernel<0>, (unsigned)blocks, threads, s, g.nt, nvec, a, o);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
