// llama_gemm_bf16_streamk_static: the stream-K tcgen05 GEMM of the decode
// projections (weights as the 128-row MMA side, a few tokens as the N side,
// K split across all SMs) with its fp32 partial sums kept in a fixed array of
// device memory owned by this library, so the call allocates nothing.
//
// Who needs this: code that cannot call cudaMalloc at the point where it runs
// the GEMM -- an engine that has already reserved all device memory for its
// own pool, or a latency-critical loop where cudaMalloc / cudaFree could
// synchronise the device -- and has no workspace to pass in.
//
// The array (kScratchBytes) is a file-scope __device__ variable: every GPU
// that loads the library holds it until the process exits.  Host code cannot
// use the variable's name as a device address (on the host it is only a
// stand-in), so the address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/llama_layer.h"
#include "gemm_tc.cuh"

namespace llama {
namespace {

constexpr size_t kScratchBytes = 16u << 20;  // 16 MiB of fp32 partial sums
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_streamk_scratch[kScratchBytes / sizeof(float)];

std::mutex g_setup_mutex;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call made with that device current).  nullptr on failure.
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_streamk_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

// D[m, n] = bf16(sum over the tile's stream-K slots of part[tile][slot][n][r])
// with m = 128 tile + r.  CTA (tile, group of 32 columns): the partials are
// read along r (their memory order), summed into shared memory and written
// along n, D's memory order.
__global__ void __launch_bounds__(256)
    streamk_reduce_kernel(const float* __restrict__ part, TcStreamK plan, int bn,
                          __nv_bfloat16* __restrict__ D, int M, int N) {
  __shared__ float s[32][129];
  const int t = blockIdx.x, n0 = blockIdx.y * 32;
  const int nseg = tc_streamk_segments(plan, t);
  const float* base = part + ((size_t)t * plan.slots * bn + n0) * 128;
  for (int e = threadIdx.x; e < 32 * 128; e += blockDim.x) {
    const int c = e >> 7, r = e & 127;
    float acc = 0.f;
    if (n0 + c < N)
      for (int j = 0; j < nseg; ++j) acc += base[(size_t)j * bn * 128 + e];
    s[c][r] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 128 * 32; e += blockDim.x) {
    const int r = e >> 5, c = e & 31;
    const int m = t * 128 + r, n = n0 + c;
    if (m < M && n < N) D[(size_t)m * N + n] = __float2bfloat16_rn(s[c][r]);
  }
}

int pick_bn(int N) { return N <= 64 ? 64 : (N <= 128 ? 128 : 256); }

}  // namespace
}  // namespace llama

using namespace llama;

extern "C" int llama_gemm_bf16_streamk_static(const void* A, const void* B,
                                              void* D, int M, int N, int K,
                                              void* stream) {
  if (!A || !B || !D || M < 0 || N < 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(A) |
                         reinterpret_cast<uintptr_t>(B) |
                         reinterpret_cast<uintptr_t>(D)) & 15u;
  if (mis) return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 8 != 0 || N > 256) return LLAMA_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return LLAMA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LLAMA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  const int bn = pick_bn(N);
  const TcStreamK plan = tc_streamk_plan(M, N, K, bn, sms);
  const size_t need = (size_t)plan.tiles * plan.slots * 128 * bn * sizeof(float);
  if (need > kScratchBytes) return LLAMA_ERR_WORKSPACE_TOO_SMALL;
  float* part = scratch_on_current_device();
  if (!part) return LLAMA_ERR_CUDA;

  CUtensorMap ta, tb;
  if (!tc_encode_bf16(&ta, A, M, K, 128) || !tc_encode_bf16(&tb, B, N, K, bn))
    return LLAMA_ERR_CUDA;
  TcEpiArgs ep;
  ep.out = part;
  ep.part_slots = plan.slots;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tc_gemm(TC_PARTIAL, bn, ta, tb, M, N, K, ep, sms, s) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  streamk_reduce_kernel<<<dim3(plan.tiles, (N + 31) / 32), 256, 0, s>>>(
      part, plan, bn, static_cast<__nv_bfloat16*>(D), M, N);
  return cudaGetLastError() == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA;
}
