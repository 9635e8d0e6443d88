// fa_check.cuh -- device-side bounds checks of the debug build.
//
// Built with -DFA_DEBUG (the debug library), each check site tests an index
// the kernel computed at run time before the access it guards: a tile
// coordinate against the tensor's extent, a ring stage against its ring (so
// a shared-memory address stays inside the CTA's window), a per-row vector
// offset against its buffer, a tensor-memory column range against the 512
// columns the CTA allocated.  A failed check records kStatusDebugCheck in the
// translation unit's status word, raises the CTA's abort flag and skips the
// access; every bounded wait of the CTA then gives up, so the CTA drains its
// copies and MMAs in flight, frees its tensor memory and exits through the
// same path as a timed-out wait.  Nothing traps.  In the product build every
// check is the constant true and generates no code.
#pragma once

#include "fa_internal.h"

namespace fa {

#ifdef FA_DEBUG
static __device__ __noinline__ bool debug_check_failed(int* status, volatile int* abort) {
    atomicCAS(status, 0, kStatusDebugCheck);
    *abort = 1;
    return false;
}
#define FA_CHECK(cond, status, abort) ((cond) ? true : ::fa::debug_check_failed((status), (abort)))
#else
#define FA_CHECK(cond, status, abort) true
#endif

}  // namespace fa
