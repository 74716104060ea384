// gcl_bounds.cuh -- index checks of the debug build.
//
// Compiled with -DGCL_DEBUG_BOUNDS, every checked global and dynamic shared-memory access
// first tests its index (or the first and last index of a strided run) against the size of
// its buffer.  An index outside records GCL_DEV_OUT_OF_BOUNDS in the device status word and
// the access is skipped (a load reads 0): no trap, no device assert, the kernel runs on and
// the host reads the status after its own synchronisation.  Without the macro the checks
// compile to `true` and cost nothing.  The helpers are host-callable so that the check
// itself is tested on the CPU.
#pragma once

#include <stdint.h>

#include "gcl.h"

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace gcl {

__host__ __device__ inline bool bounds_fail(int32_t *st) {
#ifdef __CUDA_ARCH__
    if (st != nullptr) atomicCAS(st, 0, GCL_DEV_OUT_OF_BOUNDS);
#else
    if (st != nullptr && *st == 0) *st = GCL_DEV_OUT_OF_BOUNDS;
#endif
    return false;
}

// True when every index of [lo, hi] lies in [0, n); otherwise records the failure.
__host__ __device__ inline bool range_in_bounds(int64_t lo, int64_t hi, int64_t n, int32_t *st) {
    return (lo >= 0 && hi >= lo && hi < n) ? true : bounds_fail(st);
}

}  // namespace gcl

#ifdef GCL_DEBUG_BOUNDS
#define GCL_IN_BOUNDS(i, n, st) \
    ::gcl::range_in_bounds((int64_t)(i), (int64_t)(i), (int64_t)(n), (st))
#define GCL_RANGE_IN_BOUNDS(lo, hi, n, st) \
    ::gcl::range_in_bounds((int64_t)(lo), (int64_t)(hi), (int64_t)(n), (st))
#else
#define GCL_IN_BOUNDS(i, n, st) true
#define GCL_RANGE_IN_BOUNDS(lo, hi, n, st) true
#endif
