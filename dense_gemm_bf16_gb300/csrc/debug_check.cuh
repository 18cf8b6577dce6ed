// Device-side checks of the debug build (compiled with DG_DEBUG=1 into
// libdgemm_gb300_debug.so; the product library is built without them and its
// kernels contain none of this code).
//
// A check guards one access (a global load or store, a TMA copy, a work unit
// the kernel is about to run): when its condition fails, the check sets a bit
// of the device status word that names the kind of failure and the access is
// skipped.  Nothing traps or asserts.  gemm_check_device_status reports such a
// bit as GEMM_ERR_DEVICE_CHECK.
//
// The count-writes mode (gemm_debug_count_writes) adds one to a per-element
// counter, in the caller's [batch][M][N] coordinates, at every write of an
// element's final value, so that a test can prove each output element is
// written exactly once.
#pragma once
#include <stdint.h>

#ifndef DG_DEBUG
#define DG_DEBUG 0
#endif

namespace dg {

// Status word: bit 0 a bounded wait expired; bits 8-10 a failed debug check.
enum : int {
    STATUS_TIMEOUT = 1,
    STATUS_CHECK_BOUNDS = 1 << 8,  // a global address outside its buffer
    STATUS_CHECK_UNIT = 1 << 9,    // a decoded work unit outside the problem
    STATUS_CHECK_ALIGN = 1 << 10,  // a misaligned address (shared or global)
};

#if DG_DEBUG
__device__ __forceinline__ bool dbg_ok(bool ok, int* status, int code) {
    if (!ok && status) atomicOr(status, code);
    return ok;
}
// true when the check passes; in the product build the condition is not
// even evaluated
#define DG_CHECK(cond, status, code) (::dg::dbg_ok((cond), (status), (code)))
// A wait that expired: ORed in, so that check bits set earlier survive.
#define DG_SET_TIMEOUT(status) atomicOr((status), ::dg::STATUS_TIMEOUT)
#else
#define DG_CHECK(cond, status, code) true
#define DG_SET_TIMEOUT(status) atomicExch((status), 1)
#endif

}  // namespace dg
