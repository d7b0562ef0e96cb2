// Self-test of the device-side failure path (gdn_selftest_bounded_wait).
//
// Every wait of the library's kernels on an mbarrier is bounded: after a fixed
// number of polls it gives up, the CTA frees its tensor memory, sets
// GDN_ERR_DEVICE_TIMEOUT in the workspace status word and returns, so a stuck
// copy or product becomes an error the host reads instead of a hang.  This
// kernel runs that path on purpose and safely: it allocates tensor memory, then
// waits on a barrier that nothing will ever complete (no copy, no product and
// no arrive is pending on it), with a caller-chosen poll limit, and leaves the
// way the real kernels do.  With `arrive` set, thread 0 arrives on the barrier
// first, so the same wait completes and the status word stays 0.
#include "../../include/gdn.h"
#include "kernels.h"
#include "prof.h"
#include "umma.cuh"

namespace gdn {

__global__ void __launch_bounds__(128, 1)
selftest_wait_kernel(int32_t* status, int limit, int arrive) {
    __shared__ uint64_t mbar;
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) umma::mbar_init(&mbar, 1);
    if (warp == 0) umma::tmem_alloc(&tslot, 32);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (arrive && tid == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(umma::saddr(&mbar))
                     : "memory");
    __syncthreads();
    const bool ok = __syncthreads_and(umma::mbar_wait(&mbar, 0, limit));
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tslot, 32);
    if (!ok && tid == 0) atomicExch(status, GDN_ERR_DEVICE_TIMEOUT);
}

cudaError_t launch_selftest_wait(int32_t* status, int limit, int arrive, cudaStream_t st) {
    GDN_PROF("selftest_wait", st);
    selftest_wait_kernel<<<1, 128, 0, st>>>(status, limit, arrive);
    return cudaGetLastError();
}

}  // namespace gdn

extern "C" gdn_status gdn_selftest_bounded_wait(void* ws, size_t ws_bytes, int32_t poll_limit,
                                                int32_t arrive, void* stream) {
    if (ws == nullptr || ws_bytes < sizeof(int32_t) ||
        (reinterpret_cast<uintptr_t>(ws) & 15u) != 0)
        return GDN_ERR_INVALID_ARG;
    if (poll_limit < 1 || poll_limit > (1 << 24) || (arrive != 0 && arrive != 1))
        return GDN_ERR_INVALID_ARG;
    return gdn::launch_selftest_wait(static_cast<int32_t*>(ws), poll_limit, arrive,
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}
