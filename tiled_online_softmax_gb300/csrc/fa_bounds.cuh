// fa_bounds.cuh -- bounds checks on global stores, for the checked build of libfa.
//
// Compiled with FA_DEBUG_BOUNDS defined, every kernel checks each global store's index against the
// extent of the tensor it writes before storing. A violation records the first offending site
// code and index in g_bounds_record and the store is skipped: nothing is written out of bounds,
// no trap is raised, and the host reads the record with fa_debug_bounds_report. Without the macro
// (the release build) in_bounds() is the constant true and the checks compile away.
#pragma once

#include <cstdint>

namespace fa {

enum BoundsSite : int {
    BOUNDS_FWD_O = 40,      // forward: the O tile's TMA store (first row and slice)
    BOUNDS_FWD_LSE = 41,    // forward: log-sum-exp row
    BOUNDS_FWD_PART = 42,   // forward: split partial state (o and m, l rows)
    BOUNDS_MERGE_O = 43,    // merge: output row (O and LSE)
    BOUNDS_ROPE = 44,       // rotary pass: output row and pair group
    BOUNDS_BWD_PREP = 45,   // backward preprocessing: D and base-2 LSE rows
    BOUNDS_BWD_DKDV = 46,   // backward: dK / dV rows
    BOUNDS_BWD_DQ = 47,     // backward: dQ rows
    BOUNDS_SELFTEST = 49,   // fa_debug_bounds_selftest: a planted violation
};

#ifdef FA_DEBUG_BOUNDS
constexpr bool kBoundsChecked = true;
// [0]: site code of the first violation (0: none); [1]: its index.
__device__ unsigned long long g_bounds_record[2];

__device__ __forceinline__ bool in_bounds(bool ok, int site, long long index) {
    if (ok) return true;
    if (atomicCAS(&g_bounds_record[0], 0ull, static_cast<unsigned long long>(site)) == 0ull)
        g_bounds_record[1] = static_cast<unsigned long long>(index);
    return false;
}
#else
constexpr bool kBoundsChecked = false;
__device__ __forceinline__ constexpr bool in_bounds(bool, int, long long) { return true; }
#endif

}  // namespace fa
