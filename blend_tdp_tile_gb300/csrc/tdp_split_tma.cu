// tdp_split_tma.cu -- tile split with the latent moved by the Tensor Memory Accelerator
// ("Tiled Data Parallelism (TDP)", section "What it is": the patchified latent is split
// into overlapping tiles; "Position normalization" for the positions, which the same
// CTAs split beside the copy).
//
// A unit of work is one tile-row segment: batch item b, frame f, row h and W-tile iW,
// i.e. the cells [lo_W, hi_W) of latent row (b, f, h), SW = hi_W - lo_W cells of C
// channels.  Inside every tile that holds the row (at most 2 F-tiles x 2 H-tiles,
// "combos") that segment is one contiguous run of SW*C elements of Y.  So a unit is
//   - one bulk-tensor load (cp.async.bulk.tensor.5d) of the box {C, box_w, 1, 1, 1} at
//     (0, lo_W, h, f, b) of a tensor map over this GPU's latent [B, F, H, W, C] into a
//     shared-memory stage, completing on the stage's mbarrier, and
//   - one bulk store (cp.async.bulk) of SW*C elements from the stage to each combo's
//     tile row.
// box_w is the widest W-tile; a narrower tile's box reads a few cells past its right
// edge (cells of the neighbouring segment, or the map's zero fill past W) that no
// store uses.  Consecutive units are consecutive W-tiles of one latent row, so the
// overlap cells two neighbouring segments share are read from HBM once and from L2
// the second time.
//
// Warp 0 of a CTA copies the latent; warps 1..3 split the positions of their share of
// the latent rows, a warp per row at a time, so that the positions run beside the copy
// in the same launch.  One thread drives the latent's ring of S stages: the bulk stores
// of the last PEND units stay in flight (PEND = 4, 2 or 1 by ring depth), the other
// S - PEND stages hold loads running ahead, and a stage is reloaded once the stores
// issued from it have finished reading it (cp.async.bulk.wait_group.read).  One CTA's
// ring moves about 30 GB/s, so an SM holds several: 3 CTAs with 66 KB of shared memory
// when each gets at least 64 units, else 6 with 33 KB.  Units are dealt round-robin, so
// the CTAs move through them in order together.  Every mbarrier wait has an iteration
// limit; past it the CTA records the failure in `err`, stops issuing, waits (again with
// a limit) for the loads it has in flight and for its stores, and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "tdp.h"
#include "tdp_device.cuh"
#include "tdp_internal.h"

namespace {

constexpr int kPosWarpsPerCta = 3;                 // warps of a CTA that split the positions
constexpr int kTmaThreads = 32 * (1 + kPosWarpsPerCta);   // warp 0, lane 0 drives the latent pipeline
constexpr int kTmaMaxStages = 32;
constexpr uint32_t kTmaSmemPerSm = 198u * 1024u;  // dynamic shared memory of the CTAs of one SM
constexpr uint32_t kTmaMaxBox = 256;               // tensor-map box extent limit
constexpr uint32_t kWaitRounds = 1u << 22;         // try_wait rounds before a load counts as lost
constexpr int kUnitsPerCta = 64;                   // fewer units per CTA at 3 CTAs/SM: use 6 CTAs/SM

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of the mbarrier at `bar`; false after kWaitRounds attempts.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitRounds; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t c0,
                                             int32_t c1, int32_t c2, int32_t c3, int32_t c4)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *gdst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the PEND most recent groups of bulk stores have finished reading shared memory.
template <int PEND>
__device__ __forceinline__ void bulk_wait_read_older()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(PEND) : "memory");
}

// Every bulk store of this thread is complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiles covering x along one dimension: first and (or -1) second.
__device__ __forceinline__ void cover2(const tdp_dim_geom &dg, int32_t x, int32_t &i0, int32_t &i1)
{
    const int32_t ci = (int32_t)(((uint32_t)(x + 1) * (uint32_t)dg.n + (uint32_t)(dg.L - 1)) / (uint32_t)dg.L) - 1;
    if (ci > 0 && x < dg.hi[ci - 1]) {
        i0 = ci - 1;
        i1 = ci;
    } else if (ci < dg.n - 1 && x >= dg.lo[ci + 1]) {
        i0 = ci;
        i1 = ci + 1;
    } else {
        i0 = ci;
        i1 = -1;
    }
}

struct unit_id {
    int32_t b, f, h, iW;
};

__device__ __forceinline__ unit_id unit_of(const tdp_geom &g, int64_t u)
{
    unit_id id;
    const int32_t nW = g.d[2].n;
    id.iW = (int32_t)(u % nW);
    int64_t r = u / nW;
    id.h = (int32_t)(r % g.H);
    r /= g.H;
    id.f = (int32_t)(r % g.F);
    id.b = (int32_t)(r / g.F);
    return id;
}

// Positions of one latent row (b, f, h) by one warp.  The warp first lists, in its table
// in shared memory, where the row starts in each tile holding it (per F/H combo and
// W-tile: the position-buffer index of cell w = 0, the tile's token count and, when
// normalising, the tile's mn); its lanes then stride over the row's 3*W [start, end) pairs,
// kPosBatch loads in flight each, and store every pair, minus the tile's mn when
// normalising, to each tile holding it (at most 2 x 2 x 2).
constexpr int kPosBatch = 4;

struct pos_entry {
    int64_t qpos;          // index of (d = 0, cell w = 0) of the row in the tile's positions
    int64_t Tt;            // tokens of the tile
    int32_t sub[3];        // what each dimension's pairs lose: the tile's mn, or 0
    int32_t pad;
};

__device__ __forceinline__ void split_pos_row(const tdp_geom &g, int64_t row, const int2 *__restrict__ P,
                                              int32_t normalize, int2 *__restrict__ Q,
                                              const int32_t *__restrict__ mn, pos_entry *tab, int32_t lane)
{
    const int32_t nW = g.d[2].n;
    const int32_t h = (int32_t)(row % g.H), f = (int32_t)((row / g.H) % g.F);
    const int32_t b = (int32_t)(row / ((int64_t)g.H * g.F));
    const tdp_row_combos rc = tdp_make_combos(g, f, h);
    const int64_t T = (int64_t)g.F * g.H * g.W;
    const int2 *src = P + (int64_t)b * 3 * T + ((int64_t)f * g.H + h) * g.W;
    const int32_t n = 3 * g.W;
    // the first pairs' loads in flight while the table is built
    int2 p[kPosBatch];
    auto load = [&](int32_t q0) {
#pragma unroll
        for (int u = 0; u < kPosBatch; ++u) {
            const int32_t q = q0 + 32 * u;
            if (q < n) {
                const int32_t d = q / g.W;
                p[u] = __ldcs(src + (int64_t)d * T + (q - d * g.W));
            }
        }
    };
    load(lane);
    __syncwarp();                                     // the previous row's table is no longer read
    for (int32_t e = lane; e < rc.nc * nW; e += 32) {
        const int32_t c = e / nW, iW = e - c * nW;
        const int32_t iF = rc.iF(c), iH = rc.iH(c);
        const int64_t SF = g.d[0].hi[iF] - g.d[0].lo[iF];
        const int64_t SH = g.d[1].hi[iH] - g.d[1].lo[iH];
        const int64_t SW = g.d[2].hi[iW] - g.d[2].lo[iW];
        pos_entry pe;
        pe.Tt = SF * SH * SW;
        pe.qpos = (int64_t)g.B * tdp_tile_off(g, iF, iH, iW) * 3 + (int64_t)b * 3 * pe.Tt +
                  ((int64_t)(f - g.d[0].lo[iF]) * SH + (h - g.d[1].lo[iH])) * SW - g.d[2].lo[iW];
        const int32_t tb = ((iF * g.d[1].n + iH) * nW + iW) * g.B + b;
#pragma unroll
        for (int d = 0; d < 3; ++d) pe.sub[d] = normalize ? __ldg(mn + (int64_t)tb * 3 + d) : 0;
        pe.pad = 0;
        tab[e] = pe;
    }
    __syncwarp();
    for (int32_t q0 = lane; q0 < n; q0 += 32 * kPosBatch) {
        if (q0 != lane) load(q0);
#pragma unroll
        for (int u = 0; u < kPosBatch; ++u) {
            const int32_t q = q0 + 32 * u;
            if (q >= n) break;
            const int32_t d = q / g.W, w = q - d * g.W;
            int32_t w0, w1;
            cover2(g.d[2], w, w0, w1);
            for (int32_t c = 0; c < rc.nc; ++c) {
                for (int32_t k = 0; k < 2; ++k) {
                    const int32_t iW = k ? w1 : w0;
                    if (iW < 0) break;
                    const pos_entry &pe = tab[c * nW + iW];
                    const uint32_t m = (uint32_t)pe.sub[d];
                    const int2 o = make_int2((int32_t)((uint32_t)p[u].x - m), (int32_t)((uint32_t)p[u].y - m));
                    Q[pe.qpos + (int64_t)d * pe.Tt + w] = o;
                }
            }
        }
    }
}

template <int PEND>
__global__ void __launch_bounds__(kTmaThreads)
tdp_split_tma_kernel(const __grid_constant__ CUtensorMap map, const __grid_constant__ tdp_geom g, int64_t n_units,
                     int32_t stages, uint32_t stage_stride, uint32_t box_bytes, char *__restrict__ Y,
                     int32_t *__restrict__ err, const int2 *__restrict__ P, int32_t normalize,
                     int2 *__restrict__ Q, const int32_t *__restrict__ mn)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    tdp_pdl_trigger();
    const int32_t warp = threadIdx.x >> 5;
    if (warp > 0) {
        // positions: warp w of CTA c takes rows (c * kPosWarpsPerCta + w - 1) + k * (grid x kPosWarpsPerCta)
        if (P) {
            pos_entry *tab = reinterpret_cast<pos_entry *>(dsm + (size_t)stages * (stage_stride + 8)) +
                             (warp - 1) * TDP_MAX_COMBOS * g.d[2].n;
            const int64_t rows = (int64_t)g.B * g.F * g.H;
            for (int64_t r = (int64_t)blockIdx.x * kPosWarpsPerCta + warp - 1; r < rows;
                 r += (int64_t)gridDim.x * kPosWarpsPerCta)
                split_pos_row(g, r, P, normalize, Q, mn, tab, threadIdx.x & 31);
        }
        return;
    }
    if (threadIdx.x != 0) return;
    const uint32_t stage0 = smem_addr(dsm);
    const uint32_t bar0 = stage0 + (uint32_t)stages * stage_stride;   // stages * 8 bytes of mbarriers
    for (int32_t s = 0; s < stages; ++s) mbar_init(bar0 + 8u * s);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    const int64_t n_mine = n_units > blockIdx.x ? (n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t row_bytes = (uint32_t)g.C * (uint32_t)g.esize;
    const tdp_dim_geom &dW = g.d[2];

    auto issue_load = [&](int64_t i) {
        const unit_id id = unit_of(g, blockIdx.x + i * (int64_t)gridDim.x);
        const int32_t s = (int32_t)(i % stages);
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, box_bytes);
        tma_load_box(stage0 + (uint32_t)s * stage_stride, &map, bar, 0, dW.lo[id.iW], id.h, id.f, id.b);
    };

    const int64_t pre = n_mine < stages ? n_mine : stages;
    for (int64_t i = 0; i < pre; ++i) issue_load(i);
    int64_t issued = pre;                     // loads issued so far (units 0 .. issued-1)
    int64_t lost_at = -1;                     // unit whose load did not complete in time
    for (int64_t i = 0; i < n_mine; ++i) {
        const int32_t s = (int32_t)(i % stages);
        if (!mbar_wait(bar0 + 8u * s, (uint32_t)((i / stages) & 1))) {
            lost_at = i;
            break;
        }
        // stores of unit i: one per (F, H) combo holding its row
        const unit_id id = unit_of(g, blockIdx.x + i * (int64_t)gridDim.x);
        int32_t f0, f1, h0, h1;
        cover2(g.d[0], id.f, f0, f1);
        cover2(g.d[1], id.h, h0, h1);
        const int32_t SW = dW.hi[id.iW] - dW.lo[id.iW];
        const uint32_t src = stage0 + (uint32_t)s * stage_stride;
        for (int32_t a = 0; a < 2; ++a) {
            const int32_t iF = a ? f1 : f0;
            if (iF < 0) break;
            for (int32_t e = 0; e < 2; ++e) {
                const int32_t iH = e ? h1 : h0;
                if (iH < 0) break;
                const int64_t SF = g.d[0].hi[iF] - g.d[0].lo[iF];
                const int64_t SH = g.d[1].hi[iH] - g.d[1].lo[iH];
                const int64_t Tt = SF * SH * SW;
                const int64_t tok = (int64_t)g.B * tdp_tile_off(g, iF, iH, id.iW) + (int64_t)id.b * Tt +
                                    ((int64_t)(id.f - g.d[0].lo[iF]) * SH + (id.h - g.d[1].lo[iH])) * SW;
                bulk_store(Y + tok * row_bytes, src, (uint32_t)SW * row_bytes);
            }
        }
        bulk_commit();
        // refill the stage of unit i - PEND once its stores have read it
        if (i >= PEND && issued < n_mine) {
            bulk_wait_read_older<PEND>();
            issue_load(issued);
            ++issued;
        }
    }
    if (lost_at >= 0) {
        if (err) atomicExch(err, 1);
        // let the loads still in flight (units lost_at .. issued - 1, at most one per
        // stage) land before the CTA's shared memory is released
        for (int64_t j = lost_at; j < issued; ++j) {
            const int32_t s = (int32_t)(j % stages);
            mbar_wait(bar0 + 8u * s, (uint32_t)((j / stages) & 1));
        }
    }
    bulk_wait_all();
}

// cuTensorMapEncodeTiled from the driver, looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Multiprocessors of the current device (0 on error).
int32_t device_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

template <int PEND>
cudaError_t launch_tma(unsigned grid, size_t smem, cudaStream_t s, const CUtensorMap &map, const tdp_geom &g,
                       int64_t n_units, int32_t stages, uint32_t stage_stride, uint32_t box_bytes, void *Y,
                       int32_t *err, const int32_t *P, int32_t normalize, int32_t *Q, const int32_t *mn)
{
    // raise the kernel's shared-memory limit once per device and size (not on every call, so
    // that calls after the first on a device make no attribute change, e.g. during capture)
    static std::atomic<int> raised[64];
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return ce;
    if (dev >= 64 || raised[dev].load(std::memory_order_relaxed) < (int)smem) {
        ce = cudaFuncSetAttribute(tdp_split_tma_kernel<PEND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (ce != cudaSuccess) return ce;
        if (dev < 64) {
            int cur = raised[dev].load(std::memory_order_relaxed);
            while (cur < (int)smem && !raised[dev].compare_exchange_weak(cur, (int)smem)) {
            }
        }
    }
    // a plain launch: the copy starts once all earlier work in the stream has completed
    return tdp_launch_smem(false, tdp_split_tma_kernel<PEND>, grid, kTmaThreads, smem, s, map, g, n_units, stages,
                           stage_stride, box_bytes, static_cast<char *>(Y), err, reinterpret_cast<const int2 *>(P),
                           P ? normalize : 0, reinterpret_cast<int2 *>(Q), mn);
}

}  // namespace

extern "C" tdp_status tdp_split_tma(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *mn,
                                    int32_t normalize, void *Y, int32_t *Q, int32_t *err, tdp_stream_t stream)
{
    if (!plan) return tdp_fail(TDP_ERR_INVALID_ARG, "null plan");
    const tdp_geom &g = plan->g;
    const tdp_status st = tdp_check_split_args(g, X, P, mn, normalize, Y, Q);
    if (st != TDP_OK) return st;
    if (err && !tdp_aligned(err, 4)) return tdp_fail(TDP_ERR_MISALIGNED, "err must be 4-byte aligned");
    if (g.B == 0) return tdp_ok();
    int32_t box_w = 0;
    for (int32_t i = 0; i < g.d[2].n; ++i) box_w = g.d[2].hi[i] - g.d[2].lo[i] > box_w ? g.d[2].hi[i] - g.d[2].lo[i] : box_w;
    const uint32_t box_bytes = (uint32_t)g.C * (uint32_t)box_w * (uint32_t)g.esize;
    const uint32_t stage_stride = (box_bytes + 127u) & ~127u;      // stages start 128-byte aligned
    // shared memory of a CTA: its ring of stages (+ an mbarrier each), then the row tables of
    // its position warps
    const uint32_t tables = (uint32_t)(kPosWarpsPerCta * TDP_MAX_COMBOS * g.d[2].n * sizeof(pos_entry));
    if ((uint32_t)g.C > kTmaMaxBox || (uint32_t)box_w > kTmaMaxBox ||
        2 * (stage_stride + 8) + tables > kTmaSmemPerSm / 3)
        return tdp_fail(TDP_ERR_TOO_LARGE,
                        "tdp_split_tma needs C <= 256, W-tiles at most 256 cells and two boxes of the widest "
                        "W-tile plus the position tables within 66 KB (tdp_split takes every shape)");
    PFN_cuTensorMapEncodeTiled_v12000 encode = encode_tiled();
    if (!encode) return tdp_fail(TDP_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");

    CUtensorMap map;
    const cuuint64_t dims[5] = {(cuuint64_t)g.C, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.F, (cuuint64_t)g.B};
    const cuuint64_t e = (cuuint64_t)g.esize;
    const cuuint64_t strides[4] = {e * g.C, e * g.C * g.W, e * g.C * g.W * g.H, e * g.C * g.W * g.H * g.F};
    const cuuint32_t box[5] = {(cuuint32_t)g.C, (cuuint32_t)box_w, 1, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult cr = encode(&map, g.dtype == TDP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                               5, const_cast<void *>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return tdp_fail(TDP_ERR_CUDA, "cuTensorMapEncodeTiled rejected the latent's tensor map");

    // CTAs per SM: 3 with deeper rings when every CTA has many units, else 6 (the ramp of
    // each CTA's ring then weighs more than its depth); at least two stages per CTA
    const int32_t sms = device_sms();
    if (sms <= 0) return tdp_fail(TDP_ERR_CUDA, "could not read the multiprocessor count");
    const int64_t n_units = (int64_t)g.B * g.F * g.H * g.d[2].n;
    int32_t per_sm = n_units >= (int64_t)3 * sms * kUnitsPerCta ? 3 : 6;
    if (2 * (stage_stride + 8) + tables > kTmaSmemPerSm / per_sm) per_sm = 3;
    int32_t stages = (int32_t)((kTmaSmemPerSm / per_sm - tables) / (stage_stride + 8));
    stages = stages > kTmaMaxStages ? kTmaMaxStages : stages;
    const size_t smem = (size_t)stages * (stage_stride + 8) + tables;
    const int64_t ctas = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(n_units < ctas ? n_units : ctas);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // groups of bulk stores in flight: 4, 2 or 1, leaving at least one stage to load into
    cudaError_t ce;
    if (stages > 4)
        ce = launch_tma<4>(grid, smem, s, map, g, n_units, stages, stage_stride, box_bytes, Y, err, P, normalize, Q, mn);
    else if (stages > 2)
        ce = launch_tma<2>(grid, smem, s, map, g, n_units, stages, stage_stride, box_bytes, Y, err, P, normalize, Q, mn);
    else
        ce = launch_tma<1>(grid, smem, s, map, g, n_units, stages, stage_stride, box_bytes, Y, err, P, normalize, Q, mn);
    if (ce == cudaSuccess) ce = cudaGetLastError();
    if (ce != cudaSuccess) return tdp_fail(TDP_ERR_CUDA, cudaGetErrorString(ce));
    return tdp_ok();
}
