// A 16-byte global load for data read once: through the non-coherent
// (read-only) path, not allocated in L1.  The caller guarantees the data does
// not change during the kernel and the address is 16-byte aligned.
#pragma once

#include <cstdint>

namespace {

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace
