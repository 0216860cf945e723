// selftest.cu -- exercises the kernels' failure path on purpose: one CTA
// waits, with the same bounded-wait routine every kernel uses, on an mbarrier
// that nothing will ever complete.  The wait gives up after the requested
// limit, the kernel records ATTN_ERR_TIMEOUT in the status word and returns;
// no fault, no hang, and the CUDA context stays usable.
#include "../../include/attn_gqa.h"
#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

__global__ void wait_never_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait_bounded(&bar, 0, status, &abort_flag, limit_ns);
}

}  // namespace
}  // namespace attn

extern "C" int attn_selftest_wait_timeout(uint32_t timeout_us, attn_stream_t stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return ATTN_ERR_INVALID_ARG;
  unsigned* st = attn::device_status_word();
  if (st == nullptr) return ATTN_ERR_CUDA;
  attn::wait_never_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      st, (unsigned long long)timeout_us * 1000ull);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
