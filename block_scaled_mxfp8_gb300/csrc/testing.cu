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

// Block-scaled MMA rate: one thread per CTA issues `iters` groups of four
// back-to-back MMAs of the forward's S shape (kind::mxf8f6f4, E4M3 x E4M3,
// M = 128, N = 256, K = 4 x 32, A and B K-major with the 128-byte swizzle,
// UE8M0 scales from TMEM), then waits for them; cycles[cta] = the SM clocks
// from the first issue to the completion (-1 if the bounded wait ran out).
// Operands are the E4M3 code of 1.0 with scale 1.0.  One CTA per SM (the
// dynamic shared memory keeps a second one off the SM).
constexpr int kProbeSmem = 48 * 1024 + 3 * 512 + 1024;
constexpr int kProbeDynSmem = 120 * 1024;

__global__ void __launch_bounds__(128, 1) test_mma_rate_kernel(int iters, long long* cycles, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5;
  uint8_t* sA = smem;              // 128 rows x 128 B
  uint8_t* sB = smem + 16384;      // 256 rows x 128 B
  uint8_t* sSf = smem + 49152;     // A atom, two B atoms
  for (int i = tid; i < 49152 / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
  for (int i = tid; i < 3 * 512 / 16; i += 128)
    reinterpret_cast<uint4*>(sSf)[i] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar_done, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid == 0) {
    const uint32_t tD = tmem, tSfA = tmem + 256, tSfB = tmem + 260;
    const uint64_t dSf = atom_desc(sSf);
    tmem_cp_desc(tSfA, dSf);
    tmem_cp_desc(tSfB, sdesc_adv(dSf, 512));
    tmem_cp_desc(tSfB + 4, sdesc_adv(dSf, 1024));
    const uint64_t dA = make_sdesc(smem_u32(sA), 16, 1024, kSwz128);
    const uint64_t dB = make_sdesc(smem_u32(sB), 16, 1024, kSwz128);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_mxf8_ss(tD, sdesc_adv(dA, 32 * kk), sdesc_adv(dB, 32 * kk), make_idesc_mxf8(128, 256, 0, 0, kk, kk), tSfA,
                    tSfB, (it > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit(&bar_done);
    bool ok = role_wait(&bar_done, 0, &s_abort, err, kErrTimeoutMma);
    const long long t1 = clock64();
    if (!ok) mbar_wait(&bar_done, 0, nullptr, 0);  // the MMAs must be done before the TMEM is released
    cycles[blockIdx.x] = ok ? t1 - t0 : -1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ex2 rate: sixteen warps per CTA (four per SM sub-partition, as the
// attention kernels' softmax warps), each thread running eight independent
// chains of `iters` steps x <- ex2(x) - 2 with the kernels' exponential
// (ex2.approx.ftz.f32; for x in [-2, -1] the chain stays in [-2, -1], and the
// subtraction runs on the FMA pipe); thread 0 stamps the SM clock between two
// block barriers.  One CTA per SM (the dynamic shared memory keeps a second
// one off the SM).
__global__ void __launch_bounds__(512, 1) test_ex2_rate_kernel(int iters, long long* cycles) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = -1.0f - 0.01f * static_cast<float>(threadIdx.x & 7) - 0.1f * static_cast<float>(c);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = ex2_approx(x[c]) - 2.0f;
  }
  __syncthreads();
  const long long t1 = clock64();
  const float sum = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
  if (sum > 0.0f) cycles[blockIdx.x] = -2;  // never (the chains stay negative): keeps the loop
  else if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// The forward's row maximum on full key tiles: 128 rows (one per thread, four
// warps, one TMEM lane quadrant each) of 64 fp32 values stored to TMEM, read
// back with tmem_ld32_max for columns [0, 32) and [32, 64).  out[3 r] and
// out[3 r + 1] receive the two maxima of row r, out[3 r + 2] the number of
// values that did not read back unchanged.
__global__ void __launch_bounds__(128, 1) test_tmem_max_kernel(const float* x, float* out) {
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(&s_tmem, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const float* row = x + tid * 64;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(row[c + k]);
    tmem_st8(lane_base + c, w);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  float v0[32], v1[32], m0, m1;
  tmem_ld32_max(lane_base, v0, m0);
  tmem_ld32_max(lane_base + 32, v1, m1);
  tmem_ld_wait();
  int bad = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    bad += __float_as_uint(v0[c]) != __float_as_uint(row[c]);
    bad += __float_as_uint(v1[c]) != __float_as_uint(row[32 + c]);
  }
  out[3 * tid] = m0;
  out[3 * tid + 1] = m1;
  out[3 * tid + 2] = static_cast<float>(bad);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace
}  // namespace mxa

extern "C" mxa_status mxa_test_tmem_max(const float* x, float* out, cudaStream_t stream) {
  if (!x || !out) return MXA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 3) return MXA_ERR_ALIGN;
  mxa::test_tmem_max_kernel<<<1, 128, 0, stream>>>(x, out);
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}

extern "C" mxa_status mxa_test_ex2_rate(int iters, int ctas, long long* cycles, cudaStream_t stream) {
  if (iters <= 0 || iters > (1 << 24) || ctas <= 0 || ctas > 4096 || !cycles) return MXA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(cycles) & 7) return MXA_ERR_ALIGN;
  if (cudaFuncSetAttribute(mxa::test_ex2_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           mxa::kProbeDynSmem) != cudaSuccess)
    return MXA_ERR_CUDA;
  mxa::test_ex2_rate_kernel<<<ctas, 512, mxa::kProbeDynSmem, stream>>>(iters, cycles);
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}

extern "C" mxa_status mxa_test_mma_rate(int iters, int ctas, long long* cycles, cudaStream_t stream) {
  if (iters <= 0 || iters > (1 << 24) || ctas <= 0 || ctas > 4096 || !cycles) return MXA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(cycles) & 7) return MXA_ERR_ALIGN;
  static_assert(mxa::kProbeSmem <= mxa::kProbeDynSmem, "probe operands fit the dynamic shared memory");
  int* err = mxa::device_error_word();
  if (!err) return MXA_ERR_CUDA;
  if (cudaFuncSetAttribute(mxa::test_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           mxa::kProbeDynSmem) != cudaSuccess)
    return MXA_ERR_CUDA;
  mxa::test_mma_rate_kernel<<<ctas, 128, mxa::kProbeDynSmem, stream>>>(iters, cycles, err);
  return cudaGetLastError() == cudaSuccess ? MXA_OK : MXA_ERR_CUDA;
}

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
