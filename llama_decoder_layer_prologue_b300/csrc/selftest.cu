// Self-test of the bounded waits that every pipelined kernel of the library
// relies on: a wait on an mbarrier that nothing arrives on and a wait on a
// device flag that nothing sets must each give up after the wait limit, set
// the timeout bit of a status word and return, so that the kernel ends and
// the context stays usable.  No fault, trap or endless loop is involved.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/llama_layer.h"
#include "common.cuh"

namespace llama {
namespace {

__device__ uint32_t g_never_set;   // the flag nothing sets (stays 0)
__device__ int g_selftest_out[3];  // mbarrier wait, flag wait, status word

__global__ void bounded_wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected, none will come
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    g_selftest_out[2] = 0;
    // phase 0 of a fresh barrier never completes
    const bool a = mbar_wait(&bar, 0, &g_selftest_out[2], &abort_flag);
    abort_flag = 0;  // let the second wait run to its own limit
    const bool b = flag_wait(&g_never_set, 1u, &g_selftest_out[2], &abort_flag);
    g_selftest_out[0] = a ? 1 : 0;
    g_selftest_out[1] = b ? 1 : 0;
  }
}

}  // namespace
}  // namespace llama

using namespace llama;

extern "C" int llama_selftest_bounded_waits(int observed[3], void* stream) {
  if (!observed) return LLAMA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>();
  if (cudaGetLastError() != cudaSuccess) return LLAMA_ERR_CUDA;
  int host[3] = {-1, -1, -1};
  if (cudaMemcpyFromSymbolAsync(host, g_selftest_out, sizeof(host), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  for (int i = 0; i < 3; ++i) observed[i] = host[i];
  return LLAMA_OK;
}
