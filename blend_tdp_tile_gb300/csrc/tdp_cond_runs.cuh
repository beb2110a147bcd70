// tdp_cond_runs.cuh -- the conditioning-token output reduction for up to kStageTiles
// tiles ("Tiled Data Parallelism (TDP)", section "Shared negative (reference)
// positions": a token kept by several tiles has blend weight 1/(number of tiles that
// kept it)), as a block-level routine shared by tdp_cond_blend_runs_kernel and the fused
// post-model kernel of tdp_blend_cond.
//
// A block takes kRunTok consecutive tokens of one batch item: it stages their slots
// [tile][token] in shared memory (each tile's slots are one coalesced read), lists per
// token, in ascending tile order, the rows of Ycond of the tiles that kept it, and cuts
// every list into runs of kRunRows rows.  The block's runs, token after token, are dealt
// to its lane groups (lanes across a token's channel vectors), which sum them one after
// another with no barrier in between, so a token kept by every tile (a negative-time
// token) is spread over all groups.  A token with one run is written by the group that
// summed it; the run sums of a token with more wait in shared memory and are added in
// order once per chunk of runs.  fp32 accumulation; the sum is multiplied by the token's
// weight, 1/(number of tiles that kept it (slot >= 0)) rounded once to fp32, rows at
// slot >= ncap being absent.
#pragma once

#include "tdp_device.cuh"

namespace tdp_cr {

constexpr int kStageTiles = 256;  // tiles the run kernel of the conditioning blend handles
constexpr int kRunThreads = 128;  // threads per block of the run kernel
constexpr int kRunTok = 8;        // tokens per block of the run kernel (at most 32)
constexpr int kRunMinBlocks = 8;  // resident blocks per SM the run kernel is compiled for
constexpr int kRunRows = 8;       // rows per run: a token's kept rows are summed in runs of 8
constexpr int kPartFloats = 4096; // shared-memory floats for the run sums of a chunk of runs

// a += y, 4 fp32 or 8 bf16 values; a bf16 value is added to its fp32 sum in one
// mixed-precision add (the bf16 value widened exactly, the sum rounded to nearest).
template <int BF16>
__device__ __forceinline__ void acc_add(float (&a)[8], const uint4 &y)
{
    const uint32_t w[4] = {y.x, y.y, y.z, y.w};
    if (BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            unsigned short lo, hi;
            asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w[i]));
            asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(a[2 * i]) : "h"(lo));
            asm("add.rn.f32.bf16 %0, %1, %0;" : "+f"(a[2 * i + 1]) : "h"(hi));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] += __uint_as_float(w[i]);
    }
}

// a x (1/n), the weight 1/n rounded to fp32 once, stored as 4 fp32 or 8 bf16 values.
template <int BF16>
__device__ __forceinline__ uint4 acc_weigh(const float (&a)[8], float n)
{
    const float r = __frcp_rn(n);
    if (BF16)
        return make_uint4(tdp_pack_bf16x2(a[0] * r, a[1] * r), tdp_pack_bf16x2(a[2] * r, a[3] * r),
                          tdp_pack_bf16x2(a[4] * r, a[5] * r), tdp_pack_bf16x2(a[6] * r, a[7] * r));
    return make_uint4(__float_as_uint(a[0] * r), __float_as_uint(a[1] * r), __float_as_uint(a[2] * r),
                      __float_as_uint(a[3] * r));
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

// s_slot[t][j] (row stride kRunTok + 1) = slot of token k0 + j in tile t, for tiles up to
// MAXT >= nt (-1 for tokens past N), by the whole block: thread (j, t0) loads tiles t0,
// t0 + kRunThreads / kRunTok, ..., all its loads in flight before any is stored.
template <int MAXT>
__device__ __forceinline__ void stage_slots(const int32_t *__restrict__ slot, int32_t nt, int32_t B, int32_t N,
                                            int32_t b, int32_t k0, int32_t *s_slot)
{
    constexpr int kStep = kRunThreads / kRunTok;   // tiles per pass of the block
    constexpr int kPer = MAXT / kStep;             // loads per thread
    const int32_t j = threadIdx.x % kRunTok, t0 = threadIdx.x / kRunTok;
    const bool tok_ok = k0 + j < N;
    int32_t v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int32_t t = t0 + u * kStep;
        v[u] = t < nt && tok_ok ? __ldg(slot + ((int64_t)t * B + b) * N + k0 + j) : -1;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int32_t t = t0 + u * kStep;
        if (t < nt) s_slot[t * (kRunTok + 1) + j] = v[u];
    }
}

// Block `blk` = tokens k0 .. k0 + kRunTok - 1 of batch item b (blocks numbered batch item
// after batch item), by the whole block with run_layout(nt).bytes of dynamic shared
// memory at dsm.  Waits for the work before it in the stream before it reads.
template <int BF16>
__device__ __forceinline__ void cond_runs_block(const tdp_geom &g, int32_t N, int32_t ncap, int32_t CV, int32_t lpt,
                                                const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot,
                                                uint4 *__restrict__ out, int32_t blk, unsigned char *dsm)
{
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
    const int32_t b = blk / nkb, k0 = (blk - b * nkb) * kRunTok;
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // slots of the block's tokens in every tile (each tile's are one coalesced read)
    if (nt <= kStageTiles / 2)
        stage_slots<kStageTiles / 2>(slot, nt, g.B, N, b, k0, s_slot);
    else
        stage_slots<kStageTiles>(slot, nt, g.B, N, b, k0, s_slot);
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
                               den > 0 ? acc_weigh<BF16>(part, (float)den) : make_uint4(0u, 0u, 0u, 0u));
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
                    if (act) __stcs(out + ((int64_t)b * N + k0 + j) * CV + cv, acc_weigh<BF16>(acc, (float)s_den[j]));
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

}  // namespace tdp_cr
