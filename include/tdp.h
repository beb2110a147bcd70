/*
 * tdp.h -- C ABI of the GB300 Tiled Data Parallelism (TDP) tile split / blend
 * library (libtdp.so, sm_103a).
 *
 * Source of the method: "Tiled Data Parallelism (TDP)" (LTX-2 docs,
 * multigpu).  The page's section "What it is" splits a patchified
 * (frames, height, width) latent into overlapping tiles, runs the transformer
 * per tile and blends the overlaps with trapezoidal masks that sum to one;
 * "Position normalization" shifts each tile's positions so its generated
 * tokens start at zero; "Shared negative (reference) positions" filters the
 * conditioning tokens per tile; "API / Tiling config" gives per-dimension
 * tile counts and overlaps.  On one GPU the page's cross-rank all_reduce of
 * the blended tiles becomes an on-device accumulation over all tiles.
 *
 * Conventions shared by every entry point
 *   - Dimensions are ordered (F, H, W) = (frames, height, width); d = 0 is time.
 *   - Latent X and blended Z: [B, F, H, W, C], contiguous, C fastest.
 *   - Generated-token positions P: [B, 3, T, 2] int32, T = F*H*W, token order
 *     row-major (f, h, w), last axis = [start, end).
 *   - Tiles are numbered t = (iF*nH + iH)*nW + iW; tokens inside a tile are
 *     row-major over the tile's box.  Tile t holds T_t = SF*SH*SW tokens and
 *     begins at token offset off_t = sum_{u<t} T_u (tdp_plan_info).
 *   - Tile buffers are TILE-MAJOR so that each tile's input to the per-tile
 *     transformer is one contiguous block:
 *       Y (tiles, and tile outputs Yout): tile t = contiguous [B, T_t, C] at
 *         element offset B*off_t*C;
 *       Q (tile positions): tile t = contiguous [B, 3, T_t, 2] int32 at
 *         element offset B*off_t*6.
 *   - mn, mx: [n_tiles, B, 3] int32, the minimum start and maximum end of the
 *     tile's generated-token positions (global coordinates).
 *   - Every pointer argument named "device" must be device memory of the
 *     current CUDA device; the caller allocates and owns every buffer and
 *     the stream.  The library allocates no device memory.  Latent pointers
 *     (X, Y, Yout, Z) must be 16-byte aligned and C*sizeof(element) must be a
 *     multiple of 16; int32 buffers must be 4-byte aligned, Q and P 8-byte.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     validate their arguments on the host before any launch: an invalid
 *     argument returns an error status and launches nothing.  A launch
 *     failure returns TDP_ERR_CUDA; tdp_last_error_detail() then holds the
 *     CUDA error string.  Faults inside a kernel surface on the stream's next
 *     synchronisation, as for any CUDA work.  No C++ exception crosses the ABI.
 *   - Kernels use programmatic dependent launch: a kernel may begin while the
 *     kernel before it in the stream finishes, and waits for that kernel to
 *     complete before it touches memory the kernel may write.  To the caller,
 *     stream order is that of plain launches: a call's results are visible to
 *     whatever is queued after it.
 *   - A plan is immutable once created and may be used concurrently from any
 *     number of host threads and streams.
 *   - Position arithmetic is int32 and wraps modulo 2^32.
 */
#ifndef TDP_H_
#define TDP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
struct CUstream_st;
typedef struct CUstream_st *tdp_stream_t;

typedef enum {
    TDP_OK = 0,
    TDP_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum value      */
    TDP_ERR_BAD_GEOMETRY = 2,      /* tiling not valid for the latent extent           */
    TDP_ERR_UNSUPPORTED_DTYPE = 3, /* dtype other than TDP_F32 / TDP_BF16              */
    TDP_ERR_MISALIGNED = 4,        /* C*esize % 16 != 0 or a pointer misaligned        */
    TDP_ERR_TOO_LARGE = 5,         /* beyond TDP_MAX_TILES_PER_DIM or index ranges     */
    TDP_ERR_CUDA = 6               /* a CUDA runtime / launch error                    */
} tdp_status;

typedef enum { TDP_F32 = 0, TDP_BF16 = 1 } tdp_dtype;

/* Most tiles along one dimension. */
#define TDP_MAX_TILES_PER_DIM 64

/* Per-dimension tiling: a tile COUNT and an overlap in latent grid units
 * ("API / Tiling config": DimensionTilingConfig(num_tiles, overlap)). */
typedef struct {
    int32_t num_tiles;
    int32_t overlap;
} tdp_dim_cfg;

/* One TDP problem: latent extent, channel count, storage type and the tiling
 * of (F, H, W) (the page's TileCountConfig(frames, height, width)). */
typedef struct {
    int32_t B, F, H, W, C;
    int32_t dtype;          /* tdp_dtype */
    tdp_dim_cfg dim[3];     /* F, H, W */
} tdp_problem;

typedef struct tdp_plan_s *tdp_plan_t;   /* opaque, host-owned */

/*
 * tdp_plan_create -- validate a problem and compute its tile geometry.
 * ("API / Tiling config": counts, not sizes; the box formula is not printed.)
 *
 * Boxes: along a dimension of extent L with n tiles and overlap o, the cores
 * are c_i = floor(i*L/n), i = 0..n, and tile i spans
 * [c_i - floor(o/2), c_{i+1} + (o - floor(o/2))), with no extension past 0
 * or L; neighbours overlap by exactly o cells.  Valid when 1 <= n <= L,
 * o >= 0 and, for n >= 2, floor(L/n) >= o (no cell lies in two overlaps);
 * for n = 1 the overlap is ignored.  Also checks B >= 0, C >= 1, F, H, W in
 * [1, 2^25], the dtype, C*esize % 16 == 0 and n <= TDP_MAX_TILES_PER_DIM, and
 * that the 1-D masks of every dimension sum exactly to one (integer check).
 *
 *   prob  host pointer, read only during the call.
 *   out   host pointer; receives a new plan on TDP_OK (unchanged otherwise).
 * Host only: no CUDA call.  Release with tdp_plan_destroy.
 */
tdp_status tdp_plan_create(const tdp_problem *prob, tdp_plan_t *out);

/*
 * tdp_plan_info -- read a plan's geometry (host only).
 *   n_tiles            out: number of tiles (may be NULL)
 *   total_tile_tokens  out: sum_t T_t, tokens per batch item over all tiles (may be NULL)
 *   boxes              out: [n_tiles][3][2] int32 [lo, hi) per dimension (may be NULL)
 *   offsets            out: [n_tiles + 1] int64 token offsets off_t (may be NULL)
 */
tdp_status tdp_plan_info(tdp_plan_t plan, int32_t *n_tiles, int64_t *total_tile_tokens,
                         int32_t *boxes, int64_t *offsets);

/* Release a plan (NULL is ignored).  The caller must not use it afterwards. */
void tdp_plan_destroy(tdp_plan_t plan);

/*
 * tdp_pos_bounds -- every tile's position extent: minimum start and maximum end
 * of its generated tokens, per batch item and dimension.
 * ("Position normalization": each tile's positions are shifted by the minimum
 *  start of its generated tokens, per batch item and dimension; the maximum
 *  end is the tile's far edge for the conditioning filter.)
 *
 *   P       device [B,3,T,2] int32 generated-token positions, read once.
 *   mn, mx  device [n_tiles,B,3] int32, written (global coordinates).
 *   stream  CUDA stream.
 * Positions are usually fixed by the latent grid: a caller whose positions do not
 * change between steps may compute mn/mx once and reuse them.
 */
tdp_status tdp_pos_bounds(tdp_plan_t plan, const int32_t *P, int32_t *mn, int32_t *mx,
                          tdp_stream_t stream);

/*
 * tdp_split -- tile split with tile positions and position normalisation.
 * ("What it is": split the patchified latent into tiles, each tile's tokens
 *  go to one transformer call; "Position normalization": each tile's
 *  positions are shifted by the minimum start of its generated tokens, per
 *  batch item and dimension, so they start at zero with widths kept.)
 *
 *   X          device [B,F,H,W,C] latent (dtype of the plan), read.
 *   P          device [B,3,T,2] int32 generated-token positions, read; or NULL.
 *   mn         device [n_tiles,B,3] int32 from tdp_pos_bounds, read when P is set
 *              and normalize is nonzero (may be NULL otherwise).
 *   normalize  nonzero: Q holds positions minus mn (the page's default,
 *              normalize_positions=True); zero: Q holds the global positions.
 *   Y          device tile-major tiles, B * total_tile_tokens * C elements, written.
 *   Q          device tile-major tile positions, B * total_tile_tokens * 6 int32,
 *              written; NULL exactly when P is NULL.
 *   stream     CUDA stream the work is queued on.
 * Y[t][b][j][:] = X[b, lo_F+f, lo_H+h, lo_W+w, :] for tile-local token j = (f,h,w):
 * a bit-exact copy, each latent element read once.  Buffers must not overlap.
 */
tdp_status tdp_split(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *mn, int32_t normalize,
                     void *Y, int32_t *Q, tdp_stream_t stream);

/*
 * tdp_split_tma -- tdp_split with the latent moved by the Tensor Memory Accelerator:
 * the same outputs, bit for bit.
 * ("What it is": split the patchified latent into tiles; "Position
 *  normalization": tile positions shifted by the minimum start, as in tdp_split.)
 *
 * Each tile-row segment (batch item, frame, row, W-tile) is one bulk-tensor load of a
 * box of a tensor map over X into a shared-memory stage, followed by one bulk store
 * to each tile that holds the row (the segment is contiguous in Y).  Other warps of the
 * same CTAs split the positions beside the copy.  One ordinary launch.
 *
 *   X, P, mn, normalize, Y, Q, stream   as for tdp_split.
 *   err   device int32, or NULL: set to 1 if a bulk-tensor load did not complete
 *         within the kernel's wait limit (Y is then incomplete); never cleared by the
 *         library, so the caller zeroes it.
 * Shapes: C <= 256 elements and W-tiles at most 256 cells wide (tensor-map box
 * limits), two boxes of the widest W-tile and the position tables within 66 KB of
 * shared memory; other shapes return TDP_ERR_TOO_LARGE (tdp_split takes every shape).
 * The kernel is an ordinary launch: it starts after all earlier work in the stream.
 * The first call on a device looks up the driver's tensor-map encoder and raises the
 * kernel's shared-memory limit; make it before capturing a stream into a CUDA graph.
 */
tdp_status tdp_split_tma(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *mn, int32_t normalize,
                         void *Y, int32_t *Q, int32_t *err, tdp_stream_t stream);

/*
 * tdp_norm_filter -- per-tile conditioning-token filter with normalisation.
 * ("Shared negative (reference) positions": conditioning tokens follow the
 *  generated ones; a tile keeps a token whose [start,end) interval overlaps
 *  the tile in all three dimensions, or whose time coordinate is negative;
 *  a token kept by several tiles has blend weight 1/(tiles that kept it).
 *  "Position normalization": kept tokens move by the tile's offset.)
 *
 * Tile extent in dimension d is [mn, mx) of its generated tokens; a token
 * overlaps it when [max(s,mn), min(e,mx)) is non-empty; negative time means
 * start_F < 0.  The test runs on global coordinates, per (tile, batch item).
 *
 *   K          device [B,3,N,2] int32 conditioning-token intervals, read.
 *   N          tokens per batch item (>= 0; with N = 0 only count is written, all zero).
 *   mn, mx     device [n_tiles,B,3] int32 from tdp_pos_bounds, read.
 *   normalize  nonzero: Kout = K - mn[t,b,d]; zero: Kout = K.
 *   keep       device [n_tiles,B,N] uint8, written: 1 if tile t keeps token k of item b.
 *   idx        device [n_tiles,B,N] int32, written: kept k in ascending order,
 *              then -1 up to N.
 *   count      device [n_tiles,B] int32, written: number of kept tokens.
 *   kcount     device [B,N] int32, written: number of tiles that kept token k
 *              (the denominator of the page's 1/(tiles that kept it) weight).
 *   Kout       device [n_tiles,B,3,N,2] int32: entries [t,b,d,0:count) are the
 *              kept tokens' intervals in idx order; entries past count are not written.
 *   slot       device [n_tiles,B,N] int32, or NULL: token k's position in (t,b)'s
 *              kept list, or -1 (the inverse of idx; input of tdp_cond_blend).
 *   stream     CUDA stream.
 */
tdp_status tdp_norm_filter(tdp_plan_t plan, const int32_t *K, int32_t N,
                           const int32_t *mn, const int32_t *mx, int32_t normalize,
                           uint8_t *keep, int32_t *idx, int32_t *count, int32_t *kcount,
                           int32_t *Kout, int32_t *slot, tdp_stream_t stream);

/*
 * tdp_split_filter -- the whole pre-model stage of one TDP forward in one call:
 * tdp_pos_bounds, tdp_split and tdp_norm_filter with the same arguments and
 * bit-identical results, in three launches instead of five.
 * ("What it is", "Position normalization", "Shared negative (reference)
 *  positions": split the latent into tiles, shift each tile's positions by
 *  its offset, and give each tile the conditioning tokens it keeps.)
 *
 *   X, Y, normalize     as for tdp_split.
 *   P, Q                as for tdp_split, both required (the bounds need P).
 *   mn, mx              device [n_tiles,B,3] int32, written as by tdp_pos_bounds.
 *   K, N, keep, idx, count, kcount, Kout, slot
 *                       as for tdp_norm_filter (slot may be NULL).
 *   stream              CUDA stream.
 * The copy of the latent overlaps the bounds and the filter overlaps the copy:
 * the kernels use programmatic dependent launch, ordered so that each reads
 * only what the work before it in the stream has finished writing.  Buffers
 * must not overlap one another.
 */
tdp_status tdp_split_filter(tdp_plan_t plan, const void *X, const int32_t *P, const int32_t *K, int32_t N,
                            int32_t normalize, void *Y, int32_t *Q, int32_t *mn, int32_t *mx, uint8_t *keep,
                            int32_t *idx, int32_t *count, int32_t *kcount, int32_t *Kout, int32_t *slot,
                            tdp_stream_t stream);

/*
 * tdp_cond_blend -- average each conditioning token's per-tile outputs over the
 * tiles that kept it.
 * ("Shared negative (reference) positions": a token kept by several tiles has
 *  blend weight 1/(number of tiles that kept it), so that it is not counted
 *  several times.)
 *
 * out[b,k,:] = (1/n) * sum over the tiles t that kept token k of
 * Ycond[t,b,slot[t,b,k],:], n = number of those tiles (slot >= 0, i.e. kcount);
 * one fp32 sum over those rows in ascending t, then one multiplication per element
 * by the weight 1/n (rounded once to fp32), stored in the plan's dtype.  A token
 * that no tile kept gets 0.
 *
 *   N      conditioning tokens per batch item (>= 0).
 *   ncap   rows reserved per (tile, batch item) in Ycond (>= 1).  A tile that kept
 *          the token at slot >= ncap has no stored row: its term is left out of the
 *          sum while n still counts it, so every stored term keeps the weight 1/n.
 *          ncap >= max count keeps every contribution.
 *   Ycond  device [n_tiles, B, ncap, C] (plan dtype): row p of (t,b) is the
 *          per-tile transformer's output for the p-th token t kept for item b.
 *   slot   device [n_tiles, B, N] int32 from tdp_norm_filter.
 *   out    device [B, N, C] (plan dtype), written.
 *   stream CUDA stream.
 */
tdp_status tdp_cond_blend(tdp_plan_t plan, int32_t N, int32_t ncap, const void *Ycond,
                          const int32_t *slot, void *out, tdp_stream_t stream);

/*
 * tdp_cond_records_size, tdp_cond_records, tdp_cond_blend_records -- tdp_cond_blend in two
 * parts, for a caller whose conditioning tokens stay the same from call to call (the
 * filter's slot, and so each token's rows, then do too; in a denoising loop, every step).
 * ("Shared negative (reference) positions": a token kept by several tiles has blend weight
 *  1/(number of tiles that kept it).)
 *
 * tdp_cond_records, once: the B*N tokens dealt to G = B * ceil(N/8) records of 8, so that every
 * record holds about as many rows of Ycond: tokens ranked by class of stored rows (16 classes
 * of ceil((n_tiles + 1) / 16) rows, most rows first, ties in token order), rank r at place
 * r / G of record r % G in even rounds and of record G - 1 - r % G in odd ones.  Each
 * record holds its tokens, the rows of Ycond they sum (each token's in ascending tile
 * order), the rows per token and the tiles that kept each token.
 * tdp_cond_blend_records, each call: out as tdp_cond_blend writes it, bit for bit, from the
 * records instead of the slots (each token sums its own rows, wherever it is dealt).
 *
 *   N, ncap, slot   as for tdp_cond_blend (slot from tdp_norm_filter or tdp_split_filter).
 *   recs            device int32, tdp_cond_records_size(plan, N) ints, 16-byte aligned; written
 *                   by tdp_cond_records, read by tdp_cond_blend_records.  Layout: G records of
 *                   rec = ceil4(26 + 8 * n_tiles) ints each ([0] its number, [1] its rows R,
 *                   [2..10) rows per token, [10..18) tiles that kept each token, [18..26) each
 *                   token's index b*N + k, or -1 for an empty place, [26..26+R) row numbers
 *                   (t*B + b)*ncap + slot of Ycond), then the deal (8*G ints, record after
 *                   record, token index or -1), then every token's info (8*G ints, the first
 *                   B*N used: tiles that kept it << 16 | rows stored), then every token's
 *                   stored rows in ascending tile order (B*N lists, n_tiles ints apart),
 *                   then 32 * ceil(B*N/32) + 16 ints of the deal's tables (class counts and
 *                   first ranks per 32 tokens, class offsets).
 *   Ycond, out      as for tdp_cond_blend, with the ncap the records were made with.
 * Records made for one plan, N, ncap and slot are valid only for those; a buffer that does
 * not hold them gives wrong outputs, but tdp_cond_blend_records reads no row of Ycond
 * numbered n_tiles*B*ncap or more and writes no token outside [B, N).  At most 256 tiles and
 * B*ceil(N/8)*8 below 2^31 (TDP_ERR_TOO_LARGE beyond; tdp_cond_blend takes any count).
 * tdp_cond_records runs four kernels; tdp_cond_blend_records one.
 */
tdp_status tdp_cond_records_size(tdp_plan_t plan, int32_t N, int64_t *ints);
tdp_status tdp_cond_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *slot, int32_t *recs,
                            tdp_stream_t stream);
tdp_status tdp_cond_blend_records(tdp_plan_t plan, int32_t N, int32_t ncap, const int32_t *recs, const void *Ycond,
                                  void *out, tdp_stream_t stream);

/*
 * tdp_blend_cond -- the post-model stage in one call: tdp_blend and tdp_cond_blend with
 * the same arguments and bit-identical results, in one launch instead of two.
 * ("What it is": the blended tiles are summed into the final result; "Shared negative
 *  (reference) positions": a conditioning token's outputs weigh 1/(tiles that kept it).)
 *
 *   Yout, Z                  as for tdp_blend.
 *   N, ncap, Ycond, slot, out as for tdp_cond_blend (N = 0: only the blend).
 *   stream                   CUDA stream.
 * The token blocks, latency-bound, run beside the bandwidth-bound latent rows in the
 * same grid.  With more than 256 tiles, or Ycond rows numbered past 2^32, it issues the
 * two calls one after the other.  Buffers must not overlap one another.  The first call
 * on a device raises the kernel's shared-memory limit; make it before capturing a stream
 * into a CUDA graph.
 */
tdp_status tdp_blend_cond(tdp_plan_t plan, const void *Yout, void *Z, int32_t N, int32_t ncap, const void *Ycond,
                          const int32_t *slot, void *out, tdp_stream_t stream);

/*
 * tdp_tile_mean -- mean over tiles of a per-tile untiled output (the audio path).
 * ("What it is": audio is processed untiled on every tile's forward pass and
 *  averaged across tiles; the page warns that this average is context for the
 *  video tiles, not a meaningful audio output.)
 *
 * out[b,l] = (1/n_tiles) * sum over t of A[t,b,l], fp32 accumulation: the tiles
 * of each quarter of the tile range in ascending t, then the four quarters' sums
 * in order, times the weight 1/n_tiles rounded once to fp32; stored in the plan's
 * dtype.
 *
 *   L    elements per batch item; L * sizeof(element) must be a multiple of 16.
 *   A    device [n_tiles, B, L] (plan dtype), read.
 *   out  device [B, L] (plan dtype), written.
 */
tdp_status tdp_tile_mean(tdp_plan_t plan, int64_t L, const void *A, void *out, tdp_stream_t stream);

/*
 * tdp_blend -- mask-weighted accumulation of all tile outputs into the latent.
 * ("What it is": overlapping regions are blended with trapezoidal masks and
 *  the blended tiles are summed into the final result; the masks sum to 1.
 *  The page sums ranks with one all_reduce; here every tile is on this GPU.)
 *
 * Mask of tile t at global cell (f,h,w): (r_F * r_H) * r_W, where along each
 * dimension a tile weighs 1 inside its box, except across the o-cell overlap
 * with a neighbour: with k = 0..o-1 from the overlap's left edge the right
 * tile weighs (k+1)/(o+1) and the left tile (o-k)/(o+1).  Masks are computed
 * in registers (fp32, IEEE division) and never stored.
 * Z[b,f,h,w,:] = sum over the (at most 8) tiles covering the cell, in
 * ascending t, of mask * Yout, accumulated in fp32 and stored in the plan's
 * dtype (round to nearest even).
 *
 *   Yout   device tile-major tile outputs (same layout as tdp_split's Y), read.
 *   Z      device [B,F,H,W,C] latent, written (every element).  Must not overlap Yout.
 *   stream CUDA stream.
 */
tdp_status tdp_blend(tdp_plan_t plan, const void *Yout, void *Z, tdp_stream_t stream);

/*
 * tdp_blend_partial -- one rank's share of the blend when tiles are spread over ranks
 * round-robin.
 * ("What it is": tiles are assigned to ranks round-robin, tile t to rank t % world, and
 *  a single all_reduce sums the ranks' blended tiles into the final result.)
 *
 * Zp[b,f,h,w,:] = sum over the tiles t covering the cell with t % world == rank, in
 * ascending t, of mask * Yout (the masks of tdp_blend), in fp32; +0 where the rank owns
 * no covering tile.  Summing the world ranks' Zp (the collective) and storing the sum
 * with tdp_blend_store gives the blended latent; with world == 1 this is bit for bit
 * tdp_blend.
 *
 *   rank, world  0 <= rank < world.
 *   Yout         device tile-major tile outputs in tdp_split's layout (plan dtype); only the
 *                rank's tiles are read, so the other tiles' entries need not be filled.
 *   Zp           device [B,F,H,W,C] fp32, written (every element).  Must not overlap Yout.
 *   stream       CUDA stream.
 */
tdp_status tdp_blend_partial(tdp_plan_t plan, int32_t rank, int32_t world, const void *Yout, float *Zp,
                             tdp_stream_t stream);

/*
 * tdp_blend_store -- store a summed fp32 latent (or a slab of one) in the plan's dtype.
 * ("What it is": the blended tiles, summed across ranks, are the final result.)
 *
 * Z[i] = Zsum[i] for i < n, rounded to nearest even for bf16 (a copy for fp32).
 *   n      elements; a multiple of 16 bytes of the plan's dtype (8 bf16 or 4 fp32), so
 *          any run of whole latent rows qualifies.
 *   Zsum   device fp32 [n], read.   Z  device [n] (plan dtype), written.  16-byte aligned.
 */
tdp_status tdp_blend_store(tdp_plan_t plan, int64_t n, const float *Zsum, void *Z, tdp_stream_t stream);

/*
 * Plan helpers (host only, no CUDA call).
 *
 * tdp_balanced_tile_split -- a height x width tile grid for `world` ranks
 * ("API / Usage": h_tiles, w_tiles = balanced_tile_split(world size) picks a
 * balanced 2-D spatial grid over the group; the page does not define it).
 * Reading taken: the factor pair h * w = world closest to square, h <= w
 * (video latents are wider than tall).  world >= 1.
 */
tdp_status tdp_balanced_tile_split(int32_t world, int32_t *h_tiles, int32_t *w_tiles);

/*
 * tdp_tiles_for_size -- the tile count along one dimension for a largest tile
 * size, for callers that think in sizes ("API / Tiling config" contrasts the
 * count-based TileCountConfig with the size-based VAE TilingConfig).  Returns
 * in *num_tiles the smallest valid count n (see tdp_plan_create) whose tiles
 * are all at most tile_size cells long, or TDP_ERR_BAD_GEOMETRY if none is.
 */
tdp_status tdp_tiles_for_size(int32_t L, int32_t tile_size, int32_t overlap, int32_t *num_tiles);

/*
 * tdp_rank_tiles -- the tiles rank `rank` of `world` runs under round-robin
 * assignment ("What it is": tiles are assigned round-robin, so there may be
 * more tiles than GPUs: 16 tiles on 4 GPUs is 4 tiles per rank): tile t goes
 * to rank t % world.  Writes the rank's tile ids in ascending order to `tiles`
 * (room for n_tiles, may be NULL) and their number to *n.
 */
tdp_status tdp_rank_tiles(tdp_plan_t plan, int32_t rank, int32_t world, int32_t *tiles, int32_t *n);

/* Static string naming a status. */
const char *tdp_status_str(tdp_status status);

/* Detail of the last error returned on this host thread ("" if none). */
const char *tdp_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* TDP_H_ */
