// checks.cuh -- device-side bounds checks of the W4A16_DEBUG build.
//
// Compiled with -DW4A16_DEBUG, every global store and every bulk-copy source
// range of the GEMM kernels is checked against the buffer it belongs to; a
// failed check records W4A16_ERR_BOUNDS in the device status word and the
// access is skipped -- nothing traps, so a wrong index shows up as a status
// (w4a16_device_status) and the context stays usable.  In the release build
// every check is `true` and compiles away.
#pragma once

namespace w4a16 {

constexpr unsigned int kStatusBounds = 8;  // W4A16_ERR_BOUNDS

#ifdef W4A16_DEBUG
__device__ __forceinline__ bool in_bounds(bool ok, unsigned int* status) {
    if (!ok) atomicExch(status, kStatusBounds);
    return ok;
}
#else
__device__ __forceinline__ bool in_bounds(bool, unsigned int*) { return true; }
#endif

}  // namespace w4a16
