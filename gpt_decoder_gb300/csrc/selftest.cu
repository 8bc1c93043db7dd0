// Self-test of the bounded-wait failure path shared by the tensor-core kernels.
//
// Every mbarrier wait in those kernels gives up after a time limit, records GK_ERR_TIMEOUT in
// the context's device error word, releases the tensor memory the CTA holds and returns, so a
// stalled producer ends as an error status that gk_sync reports instead of a hung GPU. This
// kernel drives that path on purpose without any fault: it allocates tensor memory, waits on an
// mbarrier that no thread arrives at (the same bounded wait, with the caller's short limit), and
// then takes the same exit the production kernels take. With `arrive` set, one thread arrives
// first and the wait succeeds: the control case.
#include "tcgen05.cuh"

namespace gk {
namespace {

using namespace tc;

constexpr int ST_THREADS = 128;
constexpr uint32_t ST_TMEM_COLS = 32;

__global__ void __launch_bounds__(ST_THREADS) wait_selftest_kernel(uint64_t limit_ns, int arrive, int* err,
                                                                   long long* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) tmem_alloc(&tmem_slot, ST_TMEM_COLS);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    const uint64_t t0 = globaltimer();
    // warp-uniform outcome, then block-wide: every thread takes the same branch below
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0, nullptr, limit_ns));
    const bool failed = __syncthreads_or(!ok) != 0;
    if (threadIdx.x == 0) {
        if (elapsed_ns) *elapsed_ns = (long long)(globaltimer() - t0);
        if (failed) report(err, GK_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_slot, ST_TMEM_COLS);
}

}  // namespace
}  // namespace gk

using namespace gk;

extern "C" gk_status gk_selftest_wait_timeout(gk_ctx* ctx, int64_t limit_ns, int arrive, long long* elapsed_ns) {
    if (!ctx) return GK_ERR_ARG;
    GK_REQUIRE(ctx, limit_ns > 0 && limit_ns <= 1000000000ll, GK_ERR_ARG,
               "gk_selftest_wait_timeout: limit must be in (0, 1 s]");
    wait_selftest_kernel<<<1, ST_THREADS, 0, ctx->stream>>>((uint64_t)limit_ns, arrive ? 1 : 0, ctx->d_err,
                                                            elapsed_ns);
    return launched(ctx, "wait_selftest");
}
