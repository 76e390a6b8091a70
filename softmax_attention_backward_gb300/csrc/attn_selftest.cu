// Self-test of the bounded waits that every kernel of the library uses on its
// pipeline mbarriers: a wait that runs out must record ATTN_DEVERR_TIMEOUT in
// the error word, raise the CTA's abort flag so that the other roles stop
// waiting, and let the CTA free its TMEM and exit normally.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {
namespace {

__global__ void __launch_bounds__(64, 1) attn_wait_selftest_kernel(int32_t* err, uint64_t limit_ns,
                                                                   int32_t* result) {
  __shared__ uint64_t bar_never, bar_other;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int s_res[2];
  __shared__ unsigned long long s_ns;
  const int warp = warp_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_never, 1);       // nothing ever arrives on either barrier
    mbar_init(&bar_other, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    // the role whose wait runs out after `limit_ns`
    AbortCtx ac{&abort_flag, err};
    ac.limit_ns = limit_ns;
    const bool done = mbar_wait(&bar_never, 0, ac);
    if (threadIdx.x == 0) s_res[0] = done ? 0 : 1;
  } else {
    // a role with the default limit: it must stop on the abort flag, long
    // before its own limit
    AbortCtx ac{&abort_flag, err};
    const uint64_t t0 = globaltimer();
    const bool done = mbar_wait(&bar_other, 0, ac);
    if (threadIdx.x == 32) {
      s_res[1] = done ? 0 : 1;
      s_ns = globaltimer() - t0;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base_sh, 32);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    int r = 0;
    if (s_res[0]) r |= 1;                                   // the short wait ran out
    if (s_res[1]) r |= 2;                                   // the other role stopped
    if (s_ns < kWaitLimitNs / 2) r |= 4;                    // ... on the abort flag
    *result = r;
  }
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_wait_selftest(int32_t* error_word, unsigned limit_us, int32_t* result,
                                            attn_stream_t stream) {
  if (!error_word || !result) return ATTN_ERR_INVALID_ARG;
  if (limit_us == 0 || limit_us > 1000000u) return ATTN_ERR_INVALID_ARG;
  attn_wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      error_word, static_cast<uint64_t>(limit_us) * 1000ull, result);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
