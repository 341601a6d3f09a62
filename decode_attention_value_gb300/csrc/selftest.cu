// selftest.cu -- an on-device check of the bounded mbarrier wait every kernel of the
// library uses: one wait on a barrier nobody arrives on (it must give up after the limit,
// set KVZ_STATUS_TIMEOUT and return) and one on a phase that is already complete (it
// must return at once).  The kernel exits normally either way; nothing faults or traps.
// Also a late writer for testing overlapped attention launches: it lets a programmatic
// dependent launch begin at once, waits a bounded time, then copies a buffer.
#include "kvz_internal.h"

namespace kvz {

__global__ void k_wait_selftest(uint64_t limit_ns, uint32_t *status, uint64_t *out)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    const uint64_t t0 = globaltimer_ns();
    const bool done = mbar_wait(b, 1u, status, limit_ns);  // phase before the first: complete
    const uint64_t t1 = globaltimer_ns();
    const bool never = mbar_wait(b, 0u, status, limit_ns);  // phase 0: no arrival ever comes
    const uint64_t t2 = globaltimer_ns();
    out[0] = t1 - t0;
    out[1] = t2 - t1;
    out[2] = (done ? 1u : 0u) | (never ? 2u : 0u);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *status, uint64_t *out, cudaStream_t stream)
{
    k_wait_selftest<<<1, 32, 0, stream>>>(limit_ns, status, out);
    return cudaGetLastError();
}

// One block: allow the dependent grid to be scheduled, wait delay_ns (globaltimer), then
// copy `words` 16-byte words from src to dst.
__global__ void k_late_writer(const uint4 *src, uint4 *dst, uint64_t words, uint64_t delay_ns)
{
    pdl_launch_dependents();
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < delay_ns) {
    }
    for (uint64_t i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
}

cudaError_t launch_late_writer(const void *src, void *dst, uint64_t bytes, uint64_t delay_ns, cudaStream_t stream)
{
    k_late_writer<<<1, 256, 0, stream>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), bytes / 16,
                                          delay_ns);
    return cudaGetLastError();
}

}  // namespace kvz
