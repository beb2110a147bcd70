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
