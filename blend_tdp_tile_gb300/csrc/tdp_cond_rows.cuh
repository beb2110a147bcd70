// tdp_cond_rows.cuh -- the conditioning-token output reduction for up to kStageTiles
// tiles ("Tiled Data Parallelism (TDP)", section "Shared negative (reference)
// positions": a token kept by several tiles has blend weight 1/(number of tiles that
// kept it)), as a block-level routine shared by tdp_cond_blend_rows_kernel and the fused
// post-model kernel of tdp_blend_cond.
//
// A block takes kTok consecutive tokens of one batch item.
//   1. Slots: the block stages the tokens' slots [tile][token] in shared memory, each
//      tile's slots one coalesced read.
//   2. Lists: a half-warp per token lists, in ascending tile order, the rows of Ycond of
//      the tiles that kept the token (lane h looks at tiles u*16 + h; ballots rank the
//      stored rows), counts the tiles that kept it, and the lists are packed into one flat
//      list, token after token.
//   3. Rows: the flat list's rows are copied into a ring of kStages shared-memory stages
//      of kChunkRows rows with cp.async, the next stage in flight while one is summed; the
//      copies of a stage are shared by all threads, so a token kept by every tile costs
//      its half-warp no more copy work than any other.
//   4. Sums: each token's half-warp adds its rows of every stage to its fp32 sums in list
//      order, so a token's sum runs over its tiles in ascending order, one row after
//      another, and does not depend on the tokens around it.  After the last stage the
//      sum is multiplied by the token's weight, 1/(number of tiles that kept it
//      (slot >= 0)) rounded once to fp32; rows at slot >= ncap are absent.
#pragma once

#include "tdp_device.cuh"

namespace tdp_cr {

constexpr int kStageTiles = 256;  // most tiles the routine handles
constexpr int kTokThreads = 128;  // threads per token block
constexpr int kTok = 8;           // tokens per block: a half-warp each
constexpr int kLanes = 16;        // lanes per token: channel vectors per slab
constexpr int kTokMinBlocks = 8;  // resident blocks per SM the token kernel is compiled for
constexpr int kChunkRows = 48;    // rows per stage of the ring
constexpr int kStages = 2;        // stages of the ring
static_assert(kTokThreads == kTok * kLanes, "a half-warp per token");
static_assert((kChunkRows * kLanes) % kTokThreads == 0, "the copies of a stage split evenly over the block");

// Bytes of a ring of kStages stages of CR rows.
__host__ __device__ constexpr size_t ring_bytes(int CR) { return (size_t)kStages * CR * kLanes * 16; }


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

// 16-byte copy global -> shared (L2 only), and its group bookkeeping.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// A block's record: what the rows and sums of its kTok tokens need, in int32 units
//   [0] block number   [1] R, its stored rows   [2, 2 + kTok) rows per token (len)
//   [2 + kTok, 2 + 2 kTok) tiles that kept each token (den)
//   [2 + 2 kTok, 2 + 3 kTok) each token's index b N + k (its output row), -1 for none
//   [kRecHead, kRecHead + R) the rows of Ycond, token after token, each token's in
//   ascending tile order (the flat list).
// It lives in shared memory while a block works, and tdp_cond_records stores one per block
// in global memory, rec_ints(nt) apart.
constexpr int kRecHead = 2 + 3 * kTok;
__host__ __device__ constexpr int64_t rec_ints(int32_t nt)
{
    return ((int64_t)kRecHead + (int64_t)kTok * nt + 3) & ~(int64_t)3;
}

// Dynamic shared memory of the routine for nt tiles and stages of CR rows (offsets in bytes):
//   ring  [kStages][CR][kLanes] uint4  row stages.  Before the rows, on the slot path, it
//         holds the staged slots [nt][kTok + 1] int32 (+1: a half-warp's column reads spread
//         over the banks) and, past them, the per-token lists [kTok][nt] uint32.
//   rec   [rec_ints(nt)] int32  the block's record
struct rows_layout {
    size_t rec, bytes;
    __host__ __device__ constexpr explicit rows_layout(int32_t nt, int CR = kChunkRows)
        : rec(ring_bytes(CR)), bytes(rec + (size_t)rec_ints(nt) * 4)
    {
    }
};
static_assert(rows_layout(kStageTiles).bytes <= 48 * 1024, "token blocks must fit the default 48 KB of shared memory");
static_assert((((size_t)kStageTiles * (kTok + 1) * 4 + 15) & ~(size_t)15) + (size_t)kStageTiles * kTok * 4 <=
                  (size_t)kStages * kChunkRows * kLanes * 16,
              "the staged slots and the per-token lists fit in the row ring");

// The tokens a block works on.  A token is its index b N + k, which is also its offset in a
// tile's slots (slot[t][b][k] = slot[t B N + b N + k]); -1 is no token.
struct block_tokens {        // tokens k0 .. k0 + kTok - 1 of batch item b (the slot path)
    int64_t base;            // b N + k0
    int32_t left;            // N - k0
    __device__ __forceinline__ int64_t tok(int32_t j) const { return j < left ? base + j : -1; }
};
struct dealt_tokens {        // tokens dealt to a record, in shared memory
    const int32_t *s;
    __device__ __forceinline__ int64_t tok(int32_t j) const { return s[j]; }
};

// s_slot[t][j] (row stride kTok + 1) = slot of token ts.tok(j) in tile t, for tiles up to
// MAXT >= nt (-1 for no token), by the whole block: thread (j, t0) loads tiles t0,
// t0 + kTokThreads / kTok, ..., all its loads in flight before any is stored (for
// consecutive tokens each warp load covers 4 tiles x 8 tokens, 4 whole 32-byte sectors).
template <int MAXT, class TS>
__device__ __forceinline__ void stage_slots(const int32_t *__restrict__ slot, int32_t nt, int64_t BN, const TS &ts,
                                            int32_t *s_slot)
{
    constexpr int kStep = kTokThreads / kTok;      // tiles per pass of the block
    constexpr int kPer = MAXT / kStep;             // loads per thread
    const int32_t j = threadIdx.x % kTok, t0 = threadIdx.x / kTok;
    const int64_t tk = ts.tok(j);
    int32_t v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int32_t t = t0 + u * kStep;
        v[u] = t < nt && tk >= 0 ? __ldg(slot + (int64_t)t * BN + tk) : -1;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int32_t t = t0 + u * kStep;
        if (t < nt) s_slot[t * (kTok + 1) + j] = v[u];
    }
}

// Token j's stored rows in ascending tile order into s_row[0 .. len), and the tiles that
// kept it (den), by its half-warp: lane h looks at tiles u*16 + h, u < NU (NU*16 >= nt);
// all of a lane's slot reads are issued before the ballots.
template <int NU>
__device__ __forceinline__ void list_rows(const int32_t *s_slot, int32_t nt, int32_t B, int32_t b, int32_t ncap,
                                          int32_t j, int32_t h, uint32_t *s_row, int32_t &len, int32_t &den)
{
    const int32_t hs = threadIdx.x & 16;                      // this half's bits in a ballot
    const uint32_t below = (1u << h) - 1u;
    int32_t sl[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int32_t t = u * kLanes + h;
        sl[u] = t < nt ? s_slot[t * (kTok + 1) + j] : -1;
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const bool st = sl[u] >= 0 && sl[u] < ncap;
        den += __popc((__ballot_sync(0xffffffffu, sl[u] >= 0) >> hs) & 0xffffu);
        const uint32_t hb = (__ballot_sync(0xffffffffu, st) >> hs) & 0xffffu;
        if (st)
            s_row[len + __popc(hb & below)] =
                ((uint32_t)(u * kLanes + h) * (uint32_t)B + (uint32_t)b) * (uint32_t)ncap + (uint32_t)sl[u];
        len += __popc(hb);
    }
}

// Token j's place in its block's flat list (thread (j, h) = (threadIdx.x / kLanes,
// threadIdx.x % kLanes)): its rows are flat[base, base + len); den tiles kept it; the block
// has R rows in all.
struct tok_rows {
    int32_t len, den, base, R;
};

// The record of block blk (tokens ts.tok(0 .. kTok - 1)) from the slots, into the record
// region `rec` of shared memory, by the whole block; ends with a barrier.
template <class TS>
__device__ __forceinline__ tok_rows rows_from_slots(const tdp_geom &g, int32_t N, int32_t ncap,
                                                    const int32_t *__restrict__ slot, int32_t blk, const TS &ts,
                                                    unsigned char *dsm, int32_t *rec)
{
    const int32_t nt = g.nt;
    const int64_t BN = (int64_t)g.B * N;
    int32_t *s_slot = reinterpret_cast<int32_t *>(dsm);
    // 1. slots
    if (nt <= kStageTiles / 2)
        stage_slots<kStageTiles / 2>(slot, nt, BN, ts, s_slot);
    else
        stage_slots<kStageTiles>(slot, nt, BN, ts, s_slot);
    __syncthreads();
    // 2. lists: half-warp j, token ts.tok(j) of batch item b; lane h looks at tiles u*16 + h,
    // so the token's stored rows come out in ascending tile order (u, then h)
    const int32_t j = threadIdx.x / kLanes, h = threadIdx.x % kLanes;
    const int64_t tk = ts.tok(j);
    const int32_t b = tk >= 0 ? (int32_t)(tk / N) : 0;
    uint32_t *s_row = reinterpret_cast<uint32_t *>(dsm + (((size_t)nt * (kTok + 1) * 4 + 15) & ~(size_t)15)) + j * nt;
    tok_rows tr;
    tr.len = 0;
    tr.den = 0;
    if (nt <= kStageTiles / 2)
        list_rows<kStageTiles / 2 / kLanes>(s_slot, nt, g.B, b, ncap, j, h, s_row, tr.len, tr.den);
    else
        list_rows<kStageTiles / kLanes>(s_slot, nt, g.B, b, ncap, j, h, s_row, tr.len, tr.den);
    if (h == 0) {
        rec[2 + j] = tr.len;
        rec[2 + kTok + j] = tr.den;
        rec[2 + 2 * kTok + j] = (int32_t)tk;
    }
    __syncthreads();
    tr.base = 0;
    tr.R = 0;
#pragma unroll
    for (int q = 0; q < kTok; ++q) {
        const int32_t lq = rec[2 + q];
        tr.base += q < j ? lq : 0;
        tr.R += lq;
    }
    uint32_t *flat = reinterpret_cast<uint32_t *>(rec + kRecHead);
    for (int32_t i = h; i < tr.len; i += kLanes) flat[tr.base + i] = s_row[i];
    if (threadIdx.x == 0) {
        rec[0] = blk;
        rec[1] = tr.R;
    }
    __syncthreads();   // the record is complete; the ring is free for the rows
    return tr;
}

// Rows and sums of a block from its record in shared memory (rec, with the flat list at
// rec + kRecHead), through a ring of stages of CR rows at dsm: the outputs of its tokens, by
// the whole block; this thread's token writes output row otok (none when otok < 0).  Rows
// numbered nrows or more are not read.
template <int BF16, int CR = kChunkRows>
__device__ __forceinline__ void rows_sum(int32_t CV, const uint4 *__restrict__ Ycond, uint4 *__restrict__ out,
                                         int64_t otok, const tok_rows &tr, unsigned char *dsm, const int32_t *rec,
                                         uint32_t nrows = 0xffffffffu)
{
    uint4 *s_ring = reinterpret_cast<uint4 *>(dsm);
    const uint32_t *s_flat = reinterpret_cast<const uint32_t *>(rec + kRecHead);
    const int32_t h = threadIdx.x % kLanes;
    const int32_t R = tr.R, base = tr.base, len = tr.len;
    static_assert((CR * kLanes) % kTokThreads == 0, "the copies of a stage split evenly over the block");
    const int32_t nslab = (CV + kLanes - 1) / kLanes;
    const bool tok_ok = otok >= 0;
    if (R == 0) {      // no stored row in the block: every output is 0
        for (int32_t cv = h; cv < CV; cv += kLanes)
            if (tok_ok) __stcs(out + otok * CV + cv, make_uint4(0u, 0u, 0u, 0u));
        return;
    }
    // 3. rows: units q = (slab of kLanes channel vectors, chunk of CR rows of the
    // flat list), copied kStages - 1 units ahead of the one being summed
    const int32_t nch = (R + CR - 1) / CR;
    const int32_t nunit = nch * nslab;
    auto issue = [&](int32_t q) {
        if (q < nunit) {
            const int32_t s = q / nch, c = q - s * nch;
            uint4 *buf = s_ring + (q % kStages) * (CR * kLanes);
#pragma unroll
            for (int i = 0; i < CR * kLanes / kTokThreads; ++i) {
                const int32_t e = threadIdx.x + i * kTokThreads;
                const int32_t fi = c * CR + e / kLanes, cv = s * kLanes + e % kLanes;
                if (fi < R && cv < CV && s_flat[fi] < nrows)
                    cp_async16(buf + e, Ycond + (uint64_t)s_flat[fi] * (uint32_t)CV + cv);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int q = 0; q < kStages - 1; ++q) issue(q);
    // 4. sums: token j's rows of each unit, in list order
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int32_t q = 0; q < nunit; ++q) {
        issue(q + kStages - 1);
        cp_async_wait<kStages - 1>();
        __syncthreads();                                      // unit q is in its stage for every thread
        const int32_t s = q / nch, c = q - s * nch;
        const int32_t cv = s * kLanes + h;
        const uint4 *buf = s_ring + (q % kStages) * (CR * kLanes);
        const int32_t i0 = max(base, c * CR), i1 = min(base + len, (c + 1) * CR);
        if (cv < CV) {
#pragma unroll 4
            for (int32_t i = i0; i < i1; ++i) acc_add<BF16>(acc, buf[(i - c * CR) * kLanes + h]);
        }
        if (c == nch - 1) {                                   // the slab's last chunk: the output
            if (tok_ok && cv < CV)
                __stcs(out + otok * CV + cv,
                       tr.den > 0 ? acc_weigh<BF16>(acc, (float)tr.den) : make_uint4(0u, 0u, 0u, 0u));
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        }
        __syncthreads();                                      // the stage may be refilled
    }
    cp_async_wait<0>();
}

// Record number i of the records tdp_cond_records stores (rec_ints(nt) ints apart from
// recs) into the record region `rec` of shared memory, by the whole block: its first
// kFirstInts ints (header and first rows) in one 16-byte load per thread, the rest once R is
// known; *blk receives its block number and *otok this thread's output token (-1 unless in
// [0, ntok)).  R and the rows per token are clamped to what a record holds, so that a record
// not made by tdp_cond_records reads and writes nothing outside its region and out.  Ends
// with a barrier.
constexpr int kFirstInts = 4 * kTokThreads;
__device__ __forceinline__ tok_rows rows_from_record(int32_t nt, int64_t ntok, const int32_t *__restrict__ recs,
                                                     int32_t i, int32_t *rec, int32_t *blk, int64_t *otok)
{
    const int64_t stride = rec_ints(nt);
    const int32_t *src = recs + (int64_t)i * stride;
    const int32_t first = stride < kFirstInts ? (int32_t)stride : kFirstInts;   // both multiples of 4
    if (4 * (int32_t)threadIdx.x < first)
        reinterpret_cast<int4 *>(rec)[threadIdx.x] = __ldg(reinterpret_cast<const int4 *>(src) + threadIdx.x);
    __syncthreads();
    *blk = rec[0];
    tok_rows tr;
    tr.R = min(max(rec[1], 0), kTok * nt);
    for (int32_t e = first + (int32_t)threadIdx.x; e < kRecHead + tr.R; e += kTokThreads) rec[e] = __ldg(src + e);
    const int32_t j = threadIdx.x / kLanes;
    tr.len = min(max(rec[2 + j], 0), nt);
    tr.den = rec[2 + kTok + j];
    const int32_t ot = rec[2 + 2 * kTok + j];
    *otok = ot >= 0 && ot < ntok ? ot : -1;
    tr.base = 0;
#pragma unroll
    for (int q = 0; q < kTok; ++q) tr.base += q < j ? min(max(rec[2 + q], 0), nt) : 0;
    __syncthreads();                                      // the whole record is in shared memory
    return tr;
}

// Block i of the per-call records path: the tokens of record i, through a ring of stages
// of CR rows (rows_layout(nt, CR).bytes of dynamic shared memory at dsm), G records and ntok
// tokens (output rows) in all, Ycond rows numbered below nrows.  Waits for the work before
// it in the stream before it reads.
template <int BF16, int CR>
__device__ __forceinline__ void cond_record_block(int32_t nt, int64_t ntok, int32_t G, uint32_t nrows, int32_t CV,
                                                  const int32_t *__restrict__ recs, const uint4 *__restrict__ Ycond,
                                                  uint4 *__restrict__ out, int32_t i, unsigned char *dsm)
{
    int32_t *rec = reinterpret_cast<int32_t *>(dsm + rows_layout(nt, CR).rec);
    tdp_pdl_trigger();
    tdp_pdl_wait();
    int32_t blk = 0;
    int64_t otok = -1;
    const tok_rows tr = rows_from_record(nt, ntok, recs, i, rec, &blk, &otok);
    if (blk < 0 || blk >= G) return;                      // not a record of this problem (block-uniform)
    rows_sum<BF16, CR>(CV, Ycond, out, otok, tr, dsm, rec, nrows);
}

// Block `blk` = tokens k0 .. k0 + kTok - 1 of batch item b (blocks numbered batch item
// after batch item), by the whole block with rows_layout(nt).bytes of dynamic shared
// memory at dsm.  Waits for the work before it in the stream before it reads.  The
// caller guarantees nt <= kStageTiles and rows of Ycond numbered below 2^32.
template <int BF16>
__device__ __forceinline__ void cond_rows_block(const tdp_geom &g, int32_t N, int32_t ncap, int32_t CV,
                                                const uint4 *__restrict__ Ycond, const int32_t *__restrict__ slot,
                                                uint4 *__restrict__ out, int32_t blk, unsigned char *dsm)
{
    int32_t *rec = reinterpret_cast<int32_t *>(dsm + rows_layout(g.nt).rec);
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t nkb = (N + kTok - 1) / kTok;
    const int32_t b = blk / nkb, k0 = (blk - b * nkb) * kTok;
    const block_tokens ts{(int64_t)b * N + k0, N - k0};
    const tok_rows tr = rows_from_slots(g, N, ncap, slot, blk, ts, dsm, rec);
    rows_sum<BF16>(CV, Ycond, out, ts.tok((int32_t)threadIdx.x / kLanes), tr, dsm, rec);
}

}  // namespace tdp_cr
