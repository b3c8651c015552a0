// testing.cu -- test hooks (include/mxa_testing.h): the device functions that
// quantize P and dS inside the attention kernels, run on caller data.
#include "../../include/mxa_testing.h"
#include "attn_common.cuh"
#include "kernels.cuh"

namespace mxa {
namespace {

__global__ void test_e4m3_kernel(const float* x, int64_t n4, uint32_t* out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(x)[i];
    out[i] = pack_e4m3x4(v.x, v.y, v.z, v.w);
  }
}

// One warp per block: lane = row, 32 values per lane (the kernels' layout).
__global__ void test_ds_kernel(const float* x, int nblocks, int shift, uint8_t* codes, uint8_t* scales) {
  const int blk = blockIdx.x;
  const int lane = threadIdx.x;
  if (blk >= nblocks) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = x[(static_cast<int64_t>(blk) * 32 + lane) * 32 + i];
  uint32_t w[8];
  const uint32_t sb = quant_ds_block32(v, shift, w);
  uint32_t* dst = reinterpret_cast<uint32_t*>(codes + (static_cast<int64_t>(blk) * 32 + lane) * 32);
#pragma unroll
  for (int k = 0; k < 8; ++k) dst[k] = w[k];
  if (lane == 0) scales[blk] = static_cast<uint8_t>(sb);
}

// One warp waits, through the kernels' own bounded wait, on an mbarrier that
// nothing arrives on.  Nothing asynchronous is in flight (no bulk copy, no
// MMA, no tensor memory), so when the budget runs out the warp records the
// error word and returns.
__global__ void test_wait_kernel(long long budget, int* err) {
  __shared__ uint64_t bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncwarp();
  role_wait(&bar, 0, &s_abort, err, kErrTimeoutOther, budget);
}

}  // namespace
}  // namespace mxa

extern "C" mxa_status mxa_test_wait_timeout(long long budget_cycles, cudaStream_t stream) {
  if (budget_cycles < 0 || budget_cycles > (1ll << 31)) return MXA_ERR_ARG;
  int* err = mxa::device_error_word();
  if (!err) return MXA_ERR_CUDA;
  mxa::test_wait_kernel<<<1, 32, 0, stream>>>(budget_cycles, err);
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}

extern "C" mxa_status mxa_test_e4m3(const float* x, int64_t n, uint8_t* codes, cudaStream_t stream) {
  if (!x || !codes || n < 0 || (n & 3)) return MXA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(codes) & 3)) return MXA_ERR_ALIGN;
  if (n == 0) return MXA_OK;
  const int64_t n4 = n / 4;
  const int blocks = static_cast<int>((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
  mxa::test_e4m3_kernel<<<blocks, 256, 0, stream>>>(x, n4, reinterpret_cast<uint32_t*>(codes));
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}

extern "C" mxa_status mxa_test_ds_blocks(const float* x, int nblocks, int shift, uint8_t* codes, uint8_t* scales,
                                         cudaStream_t stream) {
  if (!x || !codes || !scales || nblocks < 0 || shift < 0 || shift > 16) return MXA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(codes) & 3) return MXA_ERR_ALIGN;
  if (nblocks == 0) return MXA_OK;
  mxa::test_ds_kernel<<<nblocks, 32, 0, stream>>>(x, nblocks, shift, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}
