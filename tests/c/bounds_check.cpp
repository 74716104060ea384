// Host-side check of the debug build's index test (csrc/gcl_bounds.cuh): with
// GCL_DEBUG_BOUNDS an index outside its buffer is reported and records
// GCL_DEV_OUT_OF_BOUNDS (first failure only); without it the test is constant true.
#include <cstdio>

#include "gcl_bounds.cuh"

int main() {
    int32_t st = 0;
    int fails = 0;
#ifdef GCL_DEBUG_BOUNDS
    fails += !GCL_IN_BOUNDS(0, 10, &st);
    fails += !GCL_IN_BOUNDS(9, 10, &st);
    fails += !GCL_RANGE_IN_BOUNDS(2, 9, 10, &st);
    fails += st != 0;
    fails += GCL_IN_BOUNDS(10, 10, &st);             // one past the end
    fails += st != GCL_DEV_OUT_OF_BOUNDS;
    st = 0;
    fails += GCL_IN_BOUNDS(-1, 10, &st);             // negative
    fails += st != GCL_DEV_OUT_OF_BOUNDS;
    st = 0;
    fails += GCL_RANGE_IN_BOUNDS(5, 10, 10, &st);    // a strided run whose last index is out
    fails += st != GCL_DEV_OUT_OF_BOUNDS;
    st = GCL_DEV_BAD_RANGE;                          // an earlier failure is kept
    fails += GCL_IN_BOUNDS(11, 10, &st);
    fails += st != GCL_DEV_BAD_RANGE;
    fails += GCL_IN_BOUNDS((int64_t)1 << 40, (int64_t)1 << 31, nullptr);   // no status word
    std::printf("debug build: %d failures\n", fails);
#else
    fails += !GCL_IN_BOUNDS(10, 10, &st);            // compiled away: always true
    fails += st != 0;
    std::printf("release build: %d failures\n", fails);
#endif
    return fails != 0;
}
