// device_status.cuh -- device-side error reporting shared by the kernels.
//
// A plan's workspace holds a status word (bits kDevErr*) and, in status words
// 2..3, the device address of the plan's host-mapped error words (0 when there
// are none, e.g. on the allocation-free entry point). A kernel that meets an
// error sets the bit and writes a 1 into the host word of its kind (0: timeout,
// 1: internal error, 2: saturated f16 operand), so the next forward call on the
// plan reports it without synchronising (errors are returned, never trapped:
// mlxcel issue #1616, Implementation Notes).
#pragma once

#include "moe_internal.h"

namespace moe {

__device__ __forceinline__ void report_error(unsigned *status, unsigned bit) {
    atomicOr(status, bit);
    const unsigned long long host = *reinterpret_cast<volatile unsigned long long *>(status + 2);
    if (host) reinterpret_cast<volatile unsigned *>(host)[bit == kDevErrTimeout ? 0 : bit == kDevErrRange ? 2 : 1] = 1u;
}

}  // namespace moe
