// Self-test of the bounded-wait machinery: a kernel waits on an mbarrier that
// nothing ever arrives at. Every wait in the library's kernels has a time
// limit, after which the kernel records a fault bit and returns instead of
// hanging; this kernel exercises exactly that path with a short limit, so a
// test can check that the fault is reported and the context stays usable.
#include "../../include/msa.h"
#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

__global__ void wait_timeout_selftest_kernel(unsigned* fault, unsigned long long limit_ns) {
  __shared__ uint64_t never_arrives;
  if (threadIdx.x == 0) {
    mbar_init(&never_arrives, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait_for(&never_arrives, 0, fault, kFaultWaitOther, limit_ns);
}

}  // namespace
}  // namespace msa

extern "C" msa_status_t msa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return MSA_INVALID_ARG;
  unsigned* fault = msa::fault_word();
  if (fault == nullptr) return MSA_CUDA_ERROR;
  msa::wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(fault,
                                                         (unsigned long long)timeout_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_CUDA_ERROR;
}
