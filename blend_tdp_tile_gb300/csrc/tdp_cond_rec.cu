// tdp_cond_rec.cu -- the conditioning-token output reduction in two calls, for callers
// whose conditioning tokens, and so the filter's slots, stay the same from call to call
// ("Tiled Data Parallelism (TDP)", section "Shared negative (reference) positions": a token
// kept by several tiles has blend weight 1/(number of tiles that kept it)):
//   tdp_cond_records        once: the tokens dealt to blocks of kTok so that every block
//                           holds about as many rows, and every block's record
//                           (tdp_cond_rows.cuh: its tokens, their rows of Ycond, the rows
//                           per token and the tiles that kept each token);
//   tdp_cond_blend_records  each call: the outputs from the records, bit for bit those of
//                           tdp_cond_blend.
// The per-call kernel reads its block's record in one trip instead of staging the slots and
// building the lists.  A token kept by every tile holds nt rows; with blocks of consecutive
// tokens, a block holding two or three such tokens makes a long chain of ring stages that
// ends the launch.  Dealt tokens spread them over the blocks.
//
// tdp_cond_records runs four kernels:
//   tdp_cond_list_kernel   every token's stored rows of Ycond, in ascending tile order, into a
//                          list of its own (n_tiles ints apart), its stored rows and the tiles
//                          that kept it, and each block's tokens per class (a block per 32
//                          tokens, each warp over a share of the tiles, their slots read
//                          coalesced);
//   tdp_cond_scan_kernel   one block: per class of stored rows (kDealClasses classes), a scan
//                          of the list blocks' counts, and the classes' offsets (most rows
//                          first);
//   tdp_cond_walk_kernel   every token's rank (ties in token order), and rank r dealt to block
//                          snake(r mod G) (G blocks; rounds alternate direction), place r / G
//                          of its kTok;
//   tdp_cond_record_kernel every block's record, its tokens' lists copied into its flat list.
// Each token sums its own rows, in ascending tile order, wherever it is dealt: the outputs do
// not depend on the deal.
#include "tdp.h"
#include "tdp_cond_rows.cuh"
#include "tdp_internal.h"

namespace {

using namespace tdp_cr;

constexpr int kListThreads = 256;                 // 32 tokens x 8 warps
constexpr int kListWarps = kListThreads / 32;
constexpr int kDealThreads = 1024;
constexpr int kDealClasses = 16;                  // classes of stored rows the deal ranks tokens by
constexpr int kWalkThreads = 256;                 // threads per block of the deal's walk (a warp per 32 tokens)
constexpr int kScanPer = 8;                       // list blocks a lane of the deal's scan takes per pass
static_assert(kDealClasses <= 32 && kDealClasses <= kDealThreads / 32, "a lane per class, a warp per class");

// Token i = b N + k (lane i % 32 of block i / 32): warp w looks at tiles [w per, (w + 1) per),
// per = ceil(nt / 8) <= TPW.  lists[i nt .. + len) = its stored rows (t B + b) ncap + slot, in
// ascending tile order; info[i] = den << 16 | len (den: tiles with slot >= 0; len: those with
// slot < ncap); counts[c P + block] = the block's tokens of class c = min(len / width, 15)
// (P blocks).
template <int TPW>
__global__ void __launch_bounds__(kListThreads)
tdp_cond_list_kernel(int32_t nt, int32_t B, int32_t N, int32_t ncap, int32_t width, const int32_t *__restrict__ slot,
                     int32_t *__restrict__ info, uint32_t *__restrict__ lists, uint32_t *__restrict__ counts)
{
    __shared__ int32_t s_len[kListWarps][32], s_den[kListWarps][32];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int64_t ntok = (int64_t)B * N;
    const int32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t tok = (int64_t)blockIdx.x * 32 + lane;
    const bool ok = tok < ntok;
    const int32_t per = (nt + kListWarps - 1) / kListWarps;
    const int32_t t0 = w * per;
    int32_t sl[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        const int32_t t = t0 + u;
        sl[u] = ok && u < per && t < nt ? __ldg(slot + (int64_t)t * ntok + tok) : -1;
    }
    int32_t len = 0, den = 0;
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
        den += sl[u] >= 0 ? 1 : 0;
        len += sl[u] >= 0 && sl[u] < ncap ? 1 : 0;
    }
    s_len[w][lane] = len;
    s_den[w][lane] = den;
    __syncthreads();
    int32_t off = 0, L = 0, D = 0;
#pragma unroll
    for (int q = 0; q < kListWarps; ++q) {
        off += q < w ? s_len[q][lane] : 0;
        L += s_len[q][lane];
        D += s_den[q][lane];
    }
    if (w == 0) {                                         // this block's tokens per class
        const int32_t c = ok ? min(L / width, kDealClasses - 1) : -1;
        const int64_t P = (ntok + 31) / 32;
#pragma unroll
        for (int cc = 0; cc < kDealClasses; ++cc) {
            const uint32_t m = __ballot_sync(0xffffffffu, c == cc);
            if (lane == cc) counts[(int64_t)cc * P + blockIdx.x] = __popc(m);
        }
    }
    if (!ok) return;
    const uint32_t b = (uint32_t)(tok / N);
    uint32_t *dst = lists + tok * nt + off;
    int32_t c = 0;
#pragma unroll
    for (int u = 0; u < TPW; ++u)
        if (sl[u] >= 0 && sl[u] < ncap) dst[c++] = ((uint32_t)(t0 + u) * (uint32_t)B + b) * (uint32_t)ncap + (uint32_t)sl[u];
    if (w == 0) info[tok] = D << 16 | L;
}

// The deal ranks tokens by class min(len / width, kDealClasses - 1), classes in descending
// order, tokens of a class in ascending order; rank r goes to place r / G of block p = r mod G
// in even rounds, G - 1 - p in odd ones (assign[blk * kTok + q], -1 where no token goes).  The
// tokens' list blocks (32 tokens each, P of them) carry counts[c P + block] from the list
// kernel.

// One block.  Warp c: first[c P + block] = tokens of class c in the list blocks before
// `block`, 32 kScanPer blocks at a time (kScanPer consecutive blocks per lane, a shuffle scan
// of the lanes' sums, a running carry); off[c] = tokens of the classes above c.  Also empties
// every place of assign.
__global__ void __launch_bounds__(kDealThreads)
tdp_cond_scan_kernel(int64_t P, int32_t G, const uint32_t *__restrict__ counts, uint32_t *__restrict__ first,
                     uint32_t *__restrict__ off, int32_t *__restrict__ assign)
{
    __shared__ uint32_t s_tot[kDealClasses];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t i = threadIdx.x; i < (int64_t)G * kTok; i += kDealThreads) assign[i] = -1;
    if (warp < kDealClasses) {
        const uint32_t *cnt = counts + (int64_t)warp * P;
        uint32_t *fst = first + (int64_t)warp * P;
        uint32_t carry = 0;
        for (int64_t p0 = 0; p0 < P; p0 += 32 * kScanPer) {
            // lane l takes kScanPer consecutive blocks: their counts, their sum scanned over the lanes
            uint32_t v[kScanPer], sum = 0;
#pragma unroll
            for (int u = 0; u < kScanPer; ++u) {
                const int64_t p = p0 + (int64_t)lane * kScanPer + u;
                v[u] = p < P ? __ldg(cnt + p) : 0u;
                sum += v[u];
            }
            uint32_t x = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            uint32_t run = carry + x - sum;
#pragma unroll
            for (int u = 0; u < kScanPer; ++u) {
                const int64_t p = p0 + (int64_t)lane * kScanPer + u;
                if (p < P) fst[p] = run;
                run += v[u];
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_tot[warp] = carry;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t above = 0;
        for (int c = kDealClasses - 1; c >= 0; --c) {
            off[c] = above;
            above += s_tot[c];
        }
    }
}

// Warp = list block (32 tokens, a lane each): rank = off[c] + first[c P + block] + the
// block's earlier tokens of class c (a ballot), then the deal.
__global__ void __launch_bounds__(kWalkThreads)
tdp_cond_walk_kernel(int64_t ntok, int32_t G, int32_t width, const int32_t *__restrict__ info,
                     const uint32_t *__restrict__ first, const uint32_t *__restrict__ off, int32_t *__restrict__ assign)
{
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t lane = threadIdx.x & 31;
    const int64_t P = (ntok + 31) / 32;
    const int64_t pb = (int64_t)blockIdx.x * (kWalkThreads / 32) + (threadIdx.x >> 5);
    if (pb >= P) return;                                  // warp-uniform
    const int64_t i = pb * 32 + lane;
    const int32_t c = i < ntok ? min((__ldg(info + i) & 0xffff) / width, kDealClasses - 1) : -1;
    uint32_t mine = 0;
#pragma unroll
    for (int cc = 0; cc < kDealClasses; ++cc) {
        const uint32_t m = __ballot_sync(0xffffffffu, c == cc);
        if (c == cc) mine = m;
    }
    if (c < 0) return;
    const uint32_t r = __ldg(off + c) + __ldg(first + (int64_t)c * P + pb) + __popc(mine & ((1u << lane) - 1u));
    const int32_t q = (int32_t)(r / (uint32_t)G), p = (int32_t)(r - (uint32_t)q * (uint32_t)G);
    const int32_t blk = (q & 1) ? G - 1 - p : p;
    assign[(int64_t)blk * kTok + q] = (int32_t)i;
}

// The record of block blk (its tokens assign[blk * kTok .. + kTok)), stored at blk: the
// header from the tokens' info, the flat list from their lists.
__global__ void __launch_bounds__(kTokThreads)
tdp_cond_record_kernel(int32_t nt, const int32_t *__restrict__ assign, const int32_t *__restrict__ info,
                       const uint32_t *__restrict__ lists, int32_t *__restrict__ recs)
{
    __shared__ int32_t s_tok[kTok], s_len[kTok];
    tdp_pdl_trigger();
    tdp_pdl_wait();
    const int32_t blk = blockIdx.x;
    int32_t *dst = recs + (int64_t)blk * rec_ints(nt);
    if (threadIdx.x < kTok) {
        const int32_t tok = __ldg(assign + (int64_t)blk * kTok + threadIdx.x);
        const int32_t v = tok >= 0 ? __ldg(info + tok) : 0;
        s_tok[threadIdx.x] = tok;
        s_len[threadIdx.x] = v & 0xffff;
        dst[2 + threadIdx.x] = v & 0xffff;
        dst[2 + kTok + threadIdx.x] = v >> 16;
        dst[2 + 2 * kTok + threadIdx.x] = tok;
    }
    __syncthreads();
    const int32_t j = threadIdx.x / kLanes, h = threadIdx.x % kLanes;
    int32_t base = 0, R = 0;
#pragma unroll
    for (int q = 0; q < kTok; ++q) {
        base += q < j ? s_len[q] : 0;
        R += s_len[q];
    }
    const int32_t tok = s_tok[j], len = s_len[j];
    if (tok >= 0) {
        const uint32_t *src = lists + (int64_t)tok * nt;
        for (int32_t i = h; i < len; i += kLanes) dst[kRecHead + base + i] = (int32_t)__ldg(src + i);
    }
    if (threadIdx.x == 0) {
        dst[0] = blk;
        dst[1] = R;
    }
}

// Block i = record i (tdp_cond_rows.cuh's cond_record_block).
template <int BF16, int CR>
__global__ void __launch_bounds__(kTokThreads, kTokMinBlocks)
tdp_cond_blend_rec_kernel(int32_t nt, int64_t ntok, uint32_t nrows, int32_t CV, const int32_t *__restrict__ recs,
                          const uint4 *__restrict__ Ycond, uint4 *__restrict__ out)
{
    extern __shared__ __align__(16) unsigned char dsm[];
    cond_record_block<BF16, CR>(nt, ntok, (int32_t)gridDim.x, nrows, CV, recs, Ycond, out, blockIdx.x, dsm);
}

// Blocks of a problem (G = B ceil(N / kTok)); TDP_OK when the records apply.
tdp_status rec_shape(const tdp_geom &g, int32_t N, int64_t *blocks)
{
    if (N < 0) return tdp_fail(TDP_ERR_INVALID_ARG, "N must be >= 0");
    if (g.nt > kStageTiles) return tdp_fail(TDP_ERR_TOO_LARGE, "conditioning records take at most 256 tiles");
    *blocks = (int64_t)g.B * ((N + kTok - 1) / kTok);
    if (*blocks * kTok > 0x7fffffffLL) return tdp_fail(TDP_ERR_TOO_LARGE, "token indices past 2^31");
    return TDP_OK;
}

}  // namespace

extern "C" tdp_status tdp_cond_records_size(tdp_plan_t plan, int32_t N, int64_t *ints)
{
    if (!plan || !ints) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan or ints");
    int64_t G = 0;
    const tdp_status st = rec_shape(plan->g, N, &G);
    if (st != TDP_OK) return st;
    const int64_t P = ((int64_t)plan->g.B * N + 31) / 32;
    *ints = G == 0 ? 0
                   : G * rec_ints(plan->g.nt) + 2 * G * kTok + (int64_t)plan->g.B * N * plan->g.nt +
                         2 * kDealClasses * P + kDealClasses;
    return tdp_ok();
}

extern "C" tdp_status tdp_cond_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *slot, int32_t *recs,
                                       tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need ncap >= 1");
    int64_t G = 0;
    const tdp_status st = rec_shape(g, N, &G);
    if (st != TDP_OK) return st;
    if (G == 0) return tdp_ok();
    if (!slot || !recs) return tdp_fail(TDP_ERR_INVALID_ARG, "null slot or recs");
    if (!tdp_aligned(slot, 4) || !tdp_aligned(recs, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "slot needs 4-byte, recs 16-byte alignment");
    if ((uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap > 0xffffffffull)
        return tdp_fail(TDP_ERR_TOO_LARGE, "rows of Ycond numbered past 2^32");
    // after the records: the deal (kTok tokens per block), every token's info, every token's
    // list, the class counts and first ranks per list block, the classes' offsets
    const int64_t ntok = (int64_t)g.B * N;
    const int64_t P = (ntok + 31) / 32;
    int32_t *assign = recs + G * rec_ints(g.nt);
    int32_t *info = assign + G * kTok;
    uint32_t *lists = reinterpret_cast<uint32_t *>(info + G * kTok);
    uint32_t *counts = lists + ntok * g.nt;
    uint32_t *first = counts + kDealClasses * P;
    uint32_t *off = first + kDealClasses * P;
    const int32_t width = (g.nt + kDealClasses) / kDealClasses;      // rows per class: 0 .. nt in 16 classes
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = g.nt <= 16 * kListWarps
                          ? tdp_launch(true, tdp_cond_list_kernel<16>, (unsigned)P, kListThreads, s, g.nt, g.B, N,
                                       ncap, width, slot, info, lists, counts)
                          : tdp_launch(true, tdp_cond_list_kernel<kStageTiles / kListWarps>, (unsigned)P, kListThreads,
                                       s, g.nt, g.B, N, ncap, width, slot, info, lists, counts);
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_cond_scan_kernel, 1, kDealThreads, s, P, (int32_t)G,
                         static_cast<const uint32_t *>(counts), first, off, assign);
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_cond_walk_kernel, (unsigned)((P + kWalkThreads / 32 - 1) / (kWalkThreads / 32)),
                         kWalkThreads, s, ntok, (int32_t)G, width, static_cast<const int32_t *>(info),
                         static_cast<const uint32_t *>(first), static_cast<const uint32_t *>(off), assign);
    if (err == cudaSuccess)
        err = tdp_launch(true, tdp_cond_record_kernel, (unsigned)G, kTokThreads, s, g.nt,
                         static_cast<const int32_t *>(assign), static_cast<const int32_t *>(info),
                         static_cast<const uint32_t *>(lists), recs);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}

extern "C" tdp_status tdp_cond_blend_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *recs,
                                             const void *Ycond, void *out, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    if (ncap < 1) return tdp_fail(TDP_ERR_INVALID_ARG, "need ncap >= 1");
    int64_t G = 0;
    const tdp_status st = rec_shape(g, N, &G);
    if (st != TDP_OK) return st;
    if (G == 0) return tdp_ok();
    const uint64_t nrows = (uint64_t)g.nt * (uint64_t)g.B * (uint64_t)ncap;
    if (nrows > 0xffffffffull) return tdp_fail(TDP_ERR_TOO_LARGE, "rows of Ycond numbered past 2^32");
    if (!recs || !Ycond || !out) return tdp_fail(TDP_ERR_INVALID_ARG, "null recs, Ycond or out");
    if (!tdp_aligned(recs, 16) || !tdp_aligned(Ycond, 16) || !tdp_aligned(out, 16))
        return tdp_fail(TDP_ERR_MISALIGNED, "recs, Ycond and out need 16-byte alignment");
    const int32_t CV = (g.C * g.esize) >> 4;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint4 *y = reinterpret_cast<const uint4 *>(Ycond);
    uint4 *o = reinterpret_cast<uint4 *>(out);
    const size_t smem = rows_layout(g.nt).bytes;
    cudaError_t err = g.dtype == TDP_BF16
                          ? tdp_launch_smem(true, tdp_cond_blend_rec_kernel<1, kChunkRows>, (unsigned)G, kTokThreads,
                                            smem, s, g.nt, (int64_t)g.B * N, (uint32_t)nrows, CV, recs, y, o)
                          : tdp_launch_smem(true, tdp_cond_blend_rec_kernel<0, kChunkRows>, (unsigned)G, kTokThreads,
                                            smem, s, g.nt, (int64_t)g.B * N, (uint32_t)nrows, CV, recs, y, o);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(err));
    return tdp_ok();
}
