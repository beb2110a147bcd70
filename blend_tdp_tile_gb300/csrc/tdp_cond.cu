// tdp_cond.cu -- the two reductions over tiles besides the latent blend
// ("Tiled Data Parallelism (TDP)"):
//   tdp_cond_blend_runs_kernel, tdp_cond_blend_kernel
//                          each conditioning token's per-tile outputs averaged
//                          over the tiles that kept it ("Shared negative
//                          (reference) positions": weight 1/(tiles that kept it));
//   tdp_tile_mean_kernel   the audio latent averaged over all tiles ("What it
//                          is": audio is processed on every tile and averaged).
// Both are gather form and accumulate in fp32; no atomics, no scratch.  The
// conditioning blend sums each token's rows in ascending tile order in runs of
// kRunRows rows and adds the runs' sums in order; the tile mean adds the tiles of
// each quarter of the tile range in ascending order and then the four quarters'
// sums in order.
//
// tdp_cond_blend has two kernels.  With at most kStageTiles tiles (and rows of
// Ycond numbered below 2^32), tdp_cond_blend_runs_kernel gives a block kRunTok
// consecutive tokens of one batch item: it stages their slots [tile][token] in
// shared memory (each tile's slots are one coalesced read), lists per token, in
// ascending tile order, the rows of Ycond of the tiles that kept it, and cuts
// every list into runs of kRunRows rows.  The block's runs, token after token,
// are dealt to its lane groups (lanes across a token's channel vectors), which
// sum them one after another with no barrier in between, so a token kept by
// every tile (a negative-time token) is spread over all groups.  A token with
// one run is written by the group that summed it; the run sums of a token with
// more wait in shared memory and are added in order once per chunk of runs.
// With more than kStageTiles tiles, tdp_cond_blend_kernel gives each token a
// warp, which reads the token's slots 32 tiles at a time.
#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kMeanVecs = 64;     // output vectors per tile-mean block
constexpr int kMeanParts = 4;     // threads per output vector, each over a quarter of the tiles
constexpr int kMeanUnroll = 8;    // tile loads a tile-mean thread keeps in flight
constexpr int kStageTiles = 256;  // tiles the run kernel of the conditioning blend handles
constexpr int kRunThreads = 128;  // threads per block of the run kernel
constexpr int kRunTok = 8;        // tokens per block of the run kernel (at most 32)
constexpr int kRunMinBlocks = 8;  // resident blocks per SM the run kernel is compiled for
constexpr int kRunRows = 8;       // rows per run: a token's kept rows are summed in runs of 8
constexpr int kPartFloats = 4096; // shared-memory floats for the run sums of a chunk of runs

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
// up to kRowsInFlight at a time and summed in that order in runs of kRunRows,
// each run's sum added to the total when it is complete.
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
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // runs before the current one
        float run[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // the current run of kRunRows rows
        int32_t n = 0;                                       // stored rows summed so far
        int32_t den = 0;                                     // tiles that kept the token
        for (int32_t t0 = 0; t0 < g.nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < g.nt ? __ldg(slot + ((int64_t)t * g.B + b) * N + k) : -1;
            den += __popc(__ballot_sync(0xffffffffu, sl >= 0));
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
                for (int u = 0; u < kRowsInFlight; ++u) {
                    if (u < got && act) acc_add<BF16>(run, y[u]);
                    if (u < got && (n + u + 1) % kRunRows == 0) {       // a run is complete
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            acc[e] += run[e];
                            run[e] = 0.f;
                        }
                    }
                }
                n += got;
            }
        }
        if (n % kRunRows != 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += run[e];
        }
        if (act) __stcs(out + tok * CV + cv, den > 0 ? acc_div<BF16>(acc, (float)den) : make_uint4(0u, 0u, 0u, 0u));
    }
}

// Shared memory of the run kernel for nt tiles (dynamic; offsets in bytes):
//   row   [kRunTok][nt]  uint32  kept rows of Ycond per token, ascending tile
//   slot  [nt][kRunTok + 1] int32  staged slots (+1: column reads spread over the banks),
//         reused after the lists are built as part [8][P][lpt] float: run sums of a chunk
//         of P = kPartFloats / (8 lpt) runs
//   carry [2][8][32] float  sum so far of the token that continues past a chunk (by chunk parity)
//   len   [kRunTok] int32 stored rows per token, then den [kRunTok] int32 tiles that kept it
//   run0  [kRunTok + 1] int32  (first run of each token; run0[kRunTok] = runs)
//   tab   [kRunTok * ceil(nt / kRunRows)] uint16  run -> (token << 8) | run index within the token
__host__ __device__ constexpr size_t run_max(size_t a, size_t b) { return a > b ? a : b; }

struct run_layout {
    size_t slot, carry, len, run0, tab, bytes;
    __host__ __device__ constexpr explicit run_layout(int32_t nt)
        : slot((size_t)kRunTok * nt * 4),
          carry(slot + run_max((size_t)nt * (kRunTok + 1) * 4, (size_t)kPartFloats * 4)),
          len(carry + 2 * 8 * 32 * 4),
          run0(len + 2 * kRunTok * 4),
          tab(run0 + (kRunTok + 1) * 4),
          bytes((tab + (size_t)kRunTok * ((nt + kRunRows - 1) / kRunRows) * 2 + 15) & ~(size_t)15)
    {
    }
};
static_assert(run_layout(kStageTiles).bytes <= 48 * 1024, "run kernel shared memory must fit the default 48 KB");

// Sum rows i0 .. i0 + kRunRows - 1 (those below len) of a token's list into acc, in order.
template <int BF16>
__device__ __forceinline__ void run_rows(const uint32_t *rows, const uint4 *__restrict__ Ycond, int32_t CV,
                                         int32_t cv, int32_t i0, int32_t len, float (&acc)[8])
{
    uint4 y[kRunRows];
#pragma unroll
    for (int u = 0; u < kRunRows; ++u)
        if (i0 + u < len) y[u] = __ldcs(Ycond + (int64_t)rows[i0 + u] * CV + cv);
#pragma unroll
    for (int u = 0; u < kRunRows; ++u)
        if (i0 + u < len) acc_add<BF16>(acc, y[u]);
}

// Block = tokens k0 .. k0 + kRunTok - 1 of batch item b.
template <int BF16>
__global__ void __launch_bounds__(kRunThreads, kRunMinBlocks)
tdp_cond_blend_runs_kernel(const __grid_constant__ tdp_geom g, int32_t N, int32_t ncap, int32_t CV, int32_t lpt,
                           const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot,
                           uint4 *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    const int32_t nt = g.nt;
    const run_layout L(nt);
    uint32_t *s_row = reinterpret_cast<uint32_t *>(dsm);
    int32_t *s_slot = reinterpret_cast<int32_t *>(dsm + L.slot);
    float *s_part = reinterpret_cast<float *>(dsm + L.slot);
    float *s_carry = reinterpret_cast<float *>(dsm + L.carry);
    int32_t *s_len = reinterpret_cast<int32_t *>(dsm + L.len);
    int32_t *s_den = s_len + kRunTok;
    int32_t *s_run0 = reinterpret_cast<int32_t *>(dsm + L.run0);
    uint16_t *s_tab = reinterpret_cast<uint16_t *>(dsm + L.tab);
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t nkb = (N + kRunTok - 1) / kRunTok;
    const int32_t b = blockIdx.x / nkb, k0 = (blockIdx.x - b * nkb) * kRunTok;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // slots of the block's tokens in every tile (each tile's are one coalesced read),
    // all of a thread's loads in flight before any is stored
    {
        constexpr int kStep = kRunThreads / kRunTok;               // tiles per pass of the block
        constexpr int kPer = kStageTiles / kStep;                  // loads per thread
        const int32_t j = threadIdx.x % kRunTok, t0 = threadIdx.x / kRunTok;
        const bool tok_ok = k0 + j < N;
        int32_t v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int32_t t = t0 + u * kStep;
            v[u] = t < nt && tok_ok ? __ldg(slot + ((int64_t)t * g.B + b) * N + k0 + j) : -1;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int32_t t = t0 + u * kStep;
            if (t < nt) s_slot[t * (kRunTok + 1) + j] = v[u];
        }
    }
    __syncthreads();
    // per token, the rows of the tiles that kept it, in ascending tile order
    for (int32_t j = warp; j < kRunTok; j += kRunThreads / 32) {
        int32_t len = 0, den = 0;
        for (int32_t t0 = 0; t0 < nt; t0 += 32) {
            const int32_t t = t0 + lane;
            const int32_t sl = t < nt ? s_slot[t * (kRunTok + 1) + j] : -1;
            den += __popc(__ballot_sync(0xffffffffu, sl >= 0));
            const uint32_t m = __ballot_sync(0xffffffffu, sl >= 0 && sl < ncap);
            if ((m >> lane) & 1u)
                s_row[j * nt + len + __popc(m & ((1u << lane) - 1u))] = ((uint32_t)t * g.B + b) * (uint32_t)ncap + sl;
            len += __popc(m);
        }
        if (lane == 0) {
            s_len[j] = k0 + j < N ? len : -1;
            s_den[j] = den;
        }
    }
    __syncthreads();
    // runs: a token has max(1, ceil(len / kRunRows)) of them (a token no tile kept has one
    // empty run, which writes its zeros); numbered token after token
    if (warp == 0) {
        const int32_t len = lane < kRunTok ? s_len[lane] : -1;
        const int32_t nr = len < 0 ? 0 : max(1, (len + kRunRows - 1) / kRunRows);
        int32_t sc = nr;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) sc += y;
        }
        if (lane < kRunTok) s_run0[lane] = sc - nr;
        if (lane == 31) s_run0[kRunTok] = sc;
    }
    __syncthreads();
    for (int32_t j = warp; j < kRunTok; j += kRunThreads / 32) {
        const int32_t r0 = s_run0[j], nr = s_run0[j + 1] - r0;
        for (int32_t r = lane; r < nr; r += 32) s_tab[r0 + r] = (uint16_t)((j << 8) | r);
    }
    __syncthreads();
    // chunks of P runs: group q of lpt lanes sums runs c0 + q, c0 + q + G, ... one after
    // another, with no barrier between them.  A token with one run is written by its group;
    // the run sums of a token with more are kept in shared memory, and after the chunk one
    // group per such token adds them in order to the carry of the chunks before.
    const int32_t U = s_run0[kRunTok];
    const int32_t G = kRunThreads / lpt, grp = threadIdx.x / lpt, gl = threadIdx.x - grp * lpt;
    const int32_t P = kPartFloats / (8 * lpt);
    for (int32_t cv0 = 0; cv0 < CV; cv0 += lpt) {
        const int32_t cv = cv0 + gl;
        const bool act = cv < CV;
        for (int32_t c0 = 0, ci = 0; c0 < U; c0 += P, ++ci) {
            const int32_t c1 = min(U, c0 + P);
            for (int32_t u = c0 + grp; u < c1; u += G) {
                const uint32_t e = s_tab[u];
                const int32_t j = (int32_t)(e >> 8), len = s_len[j], den = s_den[j];
                float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (act) run_rows<BF16>(s_row + j * nt, Ycond, CV, cv, (int32_t)(e & 255u) * kRunRows, len, part);
                if (s_run0[j + 1] - s_run0[j] == 1) {
                    if (act)
                        __stcs(out + ((int64_t)b * N + k0 + j) * CV + cv,
                               den > 0 ? acc_div<BF16>(part, (float)den) : make_uint4(0u, 0u, 0u, 0u));
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) s_part[(x * P + (u - c0)) * lpt + gl] = part[x];
                }
            }
            __syncthreads();
            const int32_t ja = (int32_t)(s_tab[c0] >> 8), jb = (int32_t)(s_tab[c1 - 1] >> 8);
            for (int32_t j = ja + grp; j <= jb; j += G) {
                const int32_t rs = s_run0[j], re = s_run0[j + 1];
                if (re - rs <= 1) continue;
                float acc[8];
                const float *cin = s_carry + ((ci + 1) & 1) * 256;
#pragma unroll
                for (int x = 0; x < 8; ++x) acc[x] = rs < c0 ? cin[x * 32 + gl] : 0.f;
                const int32_t qe = min(re, c1);
                for (int32_t q = max(rs, c0); q < qe; ++q) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) acc[x] += s_part[(x * P + (q - c0)) * lpt + gl];
                }
                if (re <= c1) {
                    if (act) __stcs(out + ((int64_t)b * N + k0 + j) * CV + cv, acc_div<BF16>(acc, (float)s_den[j]));
                } else {
                    float *cout = s_carry + (ci & 1) * 256;
#pragma unroll
                    for (int x = 0; x < 8; ++x) cout[x * 32 + gl] = acc[x];
                }
            }
            __syncthreads();
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
        const int64_t blocks = (int64_t)g.B * ((N + kRunTok - 1) / kRunTok);
        if (blocks > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "cond blend grid too large");
        int32_t lpt = 1;                                      // lanes per token: CV rounded up to 2^k, <= 32
        while (lpt < CV && lpt < 32) lpt *= 2;
        const size_t smem = run_layout(g.nt).bytes;
        err = g.dtype == TDP_BF16
                  ? tdp_launch_smem(true, tdp_cond_blend_runs_kernel<1>, (unsigned)blocks, kRunThreads, smem, s, g, N,
                                    ncap, CV, lpt, y, slot, o)
                  : tdp_launch_smem(true, tdp_cond_blend_runs_kernel<0>, (unsigned)blocks, kRunThreads, smem, s, g, N,
                                    ncap, CV, lpt, y, slot, o);
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
