// guard.cu -- verification of the guard bands around the library's scratch.
//
// Every scratch buffer a step's kernels write (wire words or codes, M1
// partials, M1 and its reciprocal scale) is allocated with kGuardBytes of a
// fixed byte pattern directly before and directly after it.  A kernel that
// wrote past either end of its buffer would change a guard; the check runs
// when the status word is exported and records a changed guard as
// kStatusGuard in that word.  One block per guard band, one 32-bit word per
// thread; nothing is written except the status word.
#include "guard.h"

namespace lc {
namespace {

__global__ void __launch_bounds__(kGuardBytes / 4) k_guard_check(const GuardList g, int* status)
{
    const uint32_t* band = g.band[blockIdx.x];
    const uint32_t pattern = 0x01010101u * kGuardByte;
    if (band[threadIdx.x] != pattern)
        atomicOr(status, kStatusGuard);
}

}  // namespace

cudaError_t launch_guard_check(const GuardList& g, int* status, cudaStream_t s)
{
    if (g.n <= 0)
        return cudaSuccess;
    if (g.n > kMaxGuardBands || status == nullptr)
        return cudaErrorInvalidValue;
    k_guard_check<<<g.n, kGuardBytes / 4, 0, s>>>(g, status);
    return cudaGetLastError();
}

}  // namespace lc
