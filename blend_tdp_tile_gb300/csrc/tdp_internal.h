// tdp_internal.h -- host-side helpers shared by the entry points of libtdp.so.
#pragma once

#include <stdint.h>

#include "tdp_geom.h"

// Record a detail string for tdp_last_error_detail() and return `st`.
tdp_status tdp_fail(tdp_status st, const char *detail);
// Clear the detail string and return TDP_OK.
tdp_status tdp_ok();

static inline bool tdp_aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

#ifdef __CUDACC__
#include <cuda_runtime.h>

#include <utility>

// Launch `kernel` on stream `s` with `smem` bytes of dynamic shared memory; with
// `pdl` set, as a programmatic dependent launch: it may start once every block
// of the kernel before it in the stream has run griddepcontrol.launch_dependents,
// and orders its own global-memory work behind that kernel with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
static inline cudaError_t tdp_launch_smem(bool pdl, void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                          size_t smem, cudaStream_t s, Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same without dynamic shared memory.
template <typename... KArgs, typename... Args>
static inline cudaError_t tdp_launch(bool pdl, void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                     cudaStream_t s, Args &&...args)
{
    return tdp_launch_smem(pdl, kernel, grid, block, 0, s, std::forward<Args>(args)...);
}

// tdp_bounds_init_kernel (plain launch) then tdp_bounds_kernel (dependent launch)
// on stream s: mn / mx of every (tile, batch item, dim).  Arguments checked by the caller.
cudaError_t tdp_launch_bounds(const tdp_geom &g, const int32_t *P, int32_t *mn, int32_t *mx, cudaStream_t s);

// Shared argument checks of the split entry points (host only).
tdp_status tdp_check_split_args(const tdp_geom &g, const void *X, const int32_t *P, const int32_t *mn,
                                int32_t normalize, const void *Y, const int32_t *Q);
#endif
