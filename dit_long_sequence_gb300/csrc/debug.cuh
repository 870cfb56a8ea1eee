// debug.cuh -- checks and fault injection of the debug library
// (libditattn_debug.so, the same sources compiled with -DDIT_DEBUG).
//
// In the product library every helper here folds to a constant: in_bounds()
// is `true` and inject() is `false`, so the checked expressions and the
// injection branches are dead code and the kernels compile as they would
// without them.  In the debug library:
//   * in_bounds(ok, ...) records the first failed check in the device status
//     word (code DIT_ERR_BOUNDS = 6, block, role, site) and returns false, and
//     the caller skips the access it guards -- nothing out of bounds is ever
//     touched, the kernel carries on and the host reads the report;
//   * inject(a, fault, index) is true in exactly one place of one CTA: where
//     the host asked for one producer signal to be withheld (a K/V load, an
//     S commit, a P arrive), so that the roles waiting on it run into their
//     bounded waits and the whole CTA winds down.
#pragma once

#include <cstdint>

#include "internal.h"

namespace dit {

#ifdef DIT_DEBUG
constexpr bool kDebugBuild = true;
#else
constexpr bool kDebugBuild = false;
#endif

constexpr unsigned int kStatusBounds = 6u;   // DIT_ERR_BOUNDS

__device__ __forceinline__ uint32_t linear_block() {
    return blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
}

static __device__ __noinline__ void bounds_report(unsigned int* status, uint32_t role, uint32_t site) {
    if (atomicCAS(status, 0u, kStatusBounds) == 0u) {
        atomicExch(status + 1, linear_block());
        atomicExch(status + 2, role);
        atomicExch(status + 3, site);
        __threadfence();
    }
}

// True when the access guarded by `ok` may go ahead.
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* status, uint32_t role, uint32_t site) {
    if constexpr (kDebugBuild) {
        if (!ok) {
            bounds_report(status, role, site);
            return false;
        }
    }
    return true;
}

// True where the host asked this CTA to withhold signal `index` of kind `fault`.
__device__ __forceinline__ bool inject(const AttnArgs& a, uint32_t fault, int index) {
    if constexpr (kDebugBuild)
        return a.dbg_fault == fault && a.dbg_fault_index == index &&
               static_cast<int>(linear_block()) == a.dbg_fault_cta;
    return false;
}

}  // namespace dit
