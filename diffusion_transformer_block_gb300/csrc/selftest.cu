// Self-test of the bounded waits (failure detection without a GPU fault).
//
// Every wait of the tensor-core kernels goes through mbar_wait (common.cuh): it spins on
// an mbarrier phase, gives up after a time limit, sets the CTA's abort flag, records its
// site in the device error word and returns false, after which the kernel frees its
// tensor memory and returns. This kernel runs that same routine on an mbarrier that
// nothing ever arrives at, with a short limit, while holding tensor memory the way the
// real kernels do, so the give-up path, the error word and the release of tensor memory
// can be exercised on purpose. It issues no copy and no MMA, so nothing is in flight
// when the wait gives up.
#include "common.cuh"
#include "internal.h"
#include "krea_dit.h"

namespace kd {
static_assert(KREA_DIT_SITE_GEMM_PRODUCER == SITE_GEMM_PRODUCER && KREA_DIT_SITE_GEMM_MMA == SITE_GEMM_MMA &&
                  KREA_DIT_SITE_GEMM_EPILOGUE == SITE_GEMM_EPILOGUE &&
                  KREA_DIT_SITE_GEMM_TEARDOWN == SITE_GEMM_TEARDOWN && KREA_DIT_SITE_ATTN_LOAD == SITE_ATTN_LOAD &&
                  KREA_DIT_SITE_ATTN_MMA == SITE_ATTN_MMA && KREA_DIT_SITE_ATTN_SOFTMAX == SITE_ATTN_SOFTMAX &&
                  KREA_DIT_SITE_ATTN_TEARDOWN == SITE_ATTN_TEARDOWN,
              "site bits of the header and the kernels agree");

namespace {

constexpr int kSelftestThreads = 128;
constexpr uint32_t kSelftestTmemCols = 32;

__global__ void __launch_bounds__(kSelftestThreads) wait_selftest_kernel(int* err, int site, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t never;  // initialised for one arrival that never comes
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, kSelftestTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const WaitCtx wc{&abort_flag, err, limit_ns};
  mbar_wait(&never, 0, wc, site);  // gives up: phase 0 never completes
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kSelftestTmemCols);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, int site, unsigned long long limit_ns, int num_sms, cudaStream_t st) {
  if (num_sms <= 0 || !err) return cudaErrorInvalidValue;
  wait_selftest_kernel<<<num_sms, kSelftestThreads, 0, st>>>(err, site, limit_ns);
  return cudaGetLastError();
}

}  // namespace kd
