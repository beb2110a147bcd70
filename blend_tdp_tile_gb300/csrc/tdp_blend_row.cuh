// tdp_blend_row.cuh -- one latent row of the blend: mask-weighted accumulation of the
// tile outputs covering it ("Tiled Data Parallelism (TDP)", section "What it is":
// overlaps are blended with trapezoidal masks summing to one and the blended tiles are
// summed into the final result; with every tile on this GPU the page's cross-rank
// all_reduce becomes one gather pass).  Shared by tdp_blend_kernel and the fused
// post-model kernel of tdp_blend_cond.
//
// Gather form.  A block owns one latent row (b, f, h).  Once per row it builds in shared
// memory the token offsets of the row inside every covering tile (at most 2 F-tiles x
// 2 H-tiles = 4 "combos", times the W-tiles) and a table of the (at most 2) W-tiles
// covering each cell with their ramp weights.  Each output vector then sums its <= 8
// tile terms in fp32 in ascending tile order and is stored once: every tile-output byte
// is read once and every latent byte written once, with no atomics and no inter-block
// waits.  The loads in flight bound a gather, so they go through shared memory: a thread
// owns two passes of eight 16-byte slots and fills them with cp.async, issuing pass
// p + 1's copies before it sums pass p, which keeps up to 16 loads outstanding without
// holding registers.  Slot s of a pass is W-tile s & 1 of combo (s >> 1) & (nc - 1) of
// the pass's vector s >> (1 + log2 nc): 4, 2 or 1 vectors per pass for 1, 2 or 4 combos.
#pragma once

#include <stddef.h>

#include "tdp_device.cuh"

namespace tdp_bl {

constexpr int kBlendThreads = 128;
constexpr int kWTab = 1024;      // cells of the per-row W table built per pass
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

// One latent row of the blend, by the whole block (blend_smem(g) bytes of dynamic shared
// memory at dsm).  Waits for the work before it in the stream (griddepcontrol.wait)
// before it reads Yout.  PART = 0: Z holds the latent in the plan's dtype.  PART = 1, the
// round-robin partial: only the tiles t with t % world == rank are loaded and summed (the
// first of them multiplied, the others added, in the same order; +0 where the rank owns no
// covering tile), and Z holds fp32 (kElems floats per 16-byte input vector).
template <int BF16, int PART = 0>
__device__ __forceinline__ void blend_row(const tdp_geom &g, int32_t cv_shift, const uint4 *__restrict__ Yout,
                                          void *__restrict__ Zv, int32_t row, unsigned char *dsm, int32_t rank = 0,
                                          int32_t world = 1)
{
    using VM = vec_math<BF16>;
    __shared__ int64_t s_tok[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
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
    // PART: which of the row's (combo, W-tile) tiles this rank owns
    uint8_t *s_own = nullptr;
    if constexpr (PART != 0) {
        __shared__ uint8_t own_tab[TDP_MAX_COMBOS * TDP_MAX_TILES_PER_DIM];
        s_own = own_tab;
        for (int32_t e = threadIdx.x; e < nc * nW; e += blockDim.x) {
            const int32_t c = e / nW, iW = e - c * nW;
            const int32_t t = (rc.iF(c) * g.d[1].n + rc.iH(c)) * nW + iW;
            own_tab[e] = t % world == rank ? 1 : 0;
        }
        __syncthreads();
    }
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
        const int64_t zoff = ((int64_t)b * T + ((int64_t)f * g.H + h) * g.W + wbase) * CV;   // output vectors
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
                    const int32_t ce = ((sl >> 1) & (nc - 1)) * nW + iWx;
                    if (iWx >= 0 && (PART == 0 || s_own[ce]))
                        cp_async16(stage + ((buf * 8 + sl) * kBlendThreads + threadIdx.x) * 16u, ybase + s_tok[ce] + v);
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
                if constexpr (PART == 0) {
                    VM::mul(acc, rFH[0] * e.r0, sb[s0 * kBlendThreads]);          // the first term keeps the sign of zero
                    if (two) VM::fma(acc, rFH[0] * e.r1, sb[(s0 + 1) * kBlendThreads]);
#pragma unroll
                    for (int c = 1; c < TDP_MAX_COMBOS; ++c) {
                        if (c < nc) {
                            VM::fma(acc, rFH[c] * e.r0, sb[(s0 + 2 * c) * kBlendThreads]);
                            if (two) VM::fma(acc, rFH[c] * e.r1, sb[(s0 + 2 * c + 1) * kBlendThreads]);
                        }
                    }
                    __stcs(reinterpret_cast<uint4 *>(Zv) + zoff + v, VM::pack(acc));
                } else {
                    const int32_t iw0 = e.iw & 0xffff, iw1 = (e.iw >> 16) - 1;
                    bool any = false;
#pragma unroll
                    for (int c = 0; c < TDP_MAX_COMBOS; ++c) {
                        if (c < nc) {
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                if (k == 1 && !two) break;
                                if (!s_own[c * nW + (k ? iw1 : iw0)]) continue;
                                const float m = rFH[c] * (k ? e.r1 : e.r0);
                                const uint4 &y = sb[(s0 + 2 * c + k) * kBlendThreads];
                                if (!any) VM::mul(acc, m, y);                     // the first owned term
                                else VM::fma(acc, m, y);
                                any = true;
                            }
                        }
                    }
                    if (!any) {
#pragma unroll
                        for (int x = 0; x < VM::kElems; ++x) acc[x] = 0.0f;
                    }
                    float4 *dst = reinterpret_cast<float4 *>(Zv) + (zoff + v) * (VM::kElems / 4);
#pragma unroll
                    for (int x = 0; x < VM::kElems / 4; ++x)
                        __stcs(dst + x, make_float4(acc[4 * x], acc[4 * x + 1], acc[4 * x + 2], acc[4 * x + 3]));
                }
            }
        }
        __syncthreads();   // the table is rebuilt for the next cells
    }
}

// Dynamic shared memory blend_row needs: the W-cell table, then the load slots.
inline size_t blend_smem(const tdp_geom &g)
{
    return (size_t)(g.W < kWTab ? g.W : kWTab) * sizeof(tdp_wcell) + kBlendStage;
}

}  // namespace tdp_bl
