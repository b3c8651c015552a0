// attn_common.cuh -- device helpers shared by the attention kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa {

// ---- exact ceil(log2 x) helpers of the FP16 per-row dQ boost
constexpr int kCl2None = -2000;  // stands for cl2 of an all-zero operand

// cl2 of a nonzero E4M3 magnitude code (7 bits): normal codes are
// 2^(E-7) (1 + M/8), subnormal ones M 2^-9.
__device__ __forceinline__ int cl2_e4m3(uint32_t c) {
  const int E = static_cast<int>(c >> 3), M = static_cast<int>(c & 7u);
  if (E) return E - 7 + (M != 0);
  return (M <= 1 ? 0 : 32 - __clz(M - 1)) - 9;
}

// cl2 of a positive normal fp32 value
__device__ __forceinline__ int cl2_f32(float x) {
  const uint32_t u = __float_as_uint(x);
  return static_cast<int>((u >> 23) & 0xFFu) - 127 + ((u & 0x7FFFFFu) != 0);
}

// cl2 of a count n >= 1
__device__ __forceinline__ int cl2_count(int64_t n) {
  return n <= 1 ? 0 : 64 - __clzll(static_cast<unsigned long long>(n - 1));
}


// 2^x on the MUFU unit (the kernels' one exponential; the backward rebuilds P
// with the same instruction as the forward).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 values in one 64-bit register pair for the packed fp32x2 ALU
// instructions (one instruction for two elements; each lane rounds exactly as
// the scalar instruction does, so results are bit-identical).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Three-input max (one instruction for two comparisons).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Bounded wait used by every warp role: gives up after `budget` SM cycles
// (kWaitBudgetCycles in every kernel), records `code` in the device error
// word and raises the CTA's abort flag; returns early (false) once another
// role has raised it.
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          int code, long long budget = kWaitBudgetCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++it & 255u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > budget) {
        *abort_flag = 1;
        if (err) atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// Same, collective over the warp: every lane waits, and the warp continues
// only if all lanes succeeded (tcgen05.ld/st that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          int code) {
  const bool ok = role_wait(bar, parity, abort_flag, err, code);
  return __all_sync(0xffffffffu, ok);
}

// Launch order of causal work over equal documents: `groups` groups
// (document, head) of `tiles` items each, where position 0 of a group is its
// heaviest item and cost falls with the position.  Item v of the launch is
// (group, pos): group after group with positions fastest -- the CTAs running
// together share their group's tiles in L2 -- except for the last 16 groups,
// which go positions slowest, so that their heaviest items start with the
// first of them and the launch ends on short CTAs instead of the last
// groups' long ones (a list-scheduling tail of 2-3.5% of the kernel in a
// simulation of the causal B8 H32 L4096 and B4 H16 L8192 grids, 0.2-0.3%
// with this order).  32-bit: a launch holds fewer than 2^31 items.
__device__ __forceinline__ void causal_launch_order(int v, int groups, int tiles, int& group, int& pos) {
  constexpr int kTail = 16;
  const int head = groups > kTail ? groups - kTail : 0;
  const int head_items = head * tiles;
  if (v < head_items) {
    group = v / tiles;
    pos = v - group * tiles;
  } else {
    const int cnt = groups - head;
    const int idx = v - head_items;
    pos = idx / cnt;
    group = head + (idx - pos * cnt);
  }
}

// Work item of this CTA from a cost-sorted tile list: CTA i takes item i / H
// for head i % H; false when i / H is past the list's end.
__device__ __forceinline__ bool list_item(const TileItem* items, const int32_t* count, int H, int& b, int& h,
                                          int& tile, int64_t& tile_base, int64_t& other_base) {
  const int i = static_cast<int>(blockIdx.x) / H;
  h = static_cast<int>(blockIdx.x) - i * H;
  if (i >= __ldg(count)) return false;
  const int4 it = __ldg(reinterpret_cast<const int4*>(items + i));
  b = it.x;
  tile = it.y;
  tile_base = it.z;
  other_base = it.w;
  return true;
}

// One 512-byte scale atom (128 rows x 4 groups) from shared memory into 4
// TMEM columns, replicated into the four 32-lane quadrants.
__device__ __forceinline__ uint64_t atom_desc(const void* smem_atom) {
  return make_sdesc(smem_u32(smem_atom), 512, 128, kSwzNone);
}
__device__ __forceinline__ void tmem_cp_desc(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, const void* smem_atom) {
  tmem_cp_desc(taddr, atom_desc(smem_atom));
}

// A shared-memory descriptor advanced by `bytes` (a multiple of 16): only the
// start-address field (bits 0-13, in 16-byte units) changes, and the kernels
// keep every operand below 256 KB so the field never carries.  The MMA
// issuers build their descriptors once and step them with this, keeping the
// single issuing thread's work per MMA to a few integer adds.
__device__ __forceinline__ uint64_t sdesc_adv(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// First scale tile of document b: sum over earlier documents of ceil(n / 128).
// Called by every thread of the CTA.
__device__ __forceinline__ int64_t doc_tile_base(const int32_t* cu, int b, int64_t len, int tid, int nthreads,
                                                 int64_t* s_slot) {
  if (cu == nullptr) return static_cast<int64_t>(b) * ((len + 127) / 128);
  if (tid == 0) *s_slot = 0;
  __syncthreads();
  int64_t part = 0;
  for (int i = tid; i < b; i += nthreads) part += (cu[i + 1] - cu[i] + 127) / 128;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((tid & 31) == 0 && part)
    atomicAdd(reinterpret_cast<unsigned long long*>(s_slot), static_cast<unsigned long long>(part));
  __syncthreads();
  return *s_slot;
}

// Two E4M3 codes (low 16 bits) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two_codes)));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace mxa

namespace mxa {

// Quantize one 32 x 32 dS block held as 32 values per lane across a warp
// (lane = row): block max-abs by a warp reduction in this register layout (no
// transpose), exponent e = ceil(log2(amax / 448)) shifted down by `shift` when
// the values carry a 2^shift boost and floored at the UE8M0 minimum, E4M3
// codes of x * 2^-(e + shift) into w.  Returns the UE8M0 byte of e.
__device__ __forceinline__ uint32_t quant_ds_block32(const float (&x)[32], int shift, uint32_t (&w)[8]) {
  // max-abs in four independent chains of three-input max
  float m0 = fmax3(fabsf(x[0]), fabsf(x[1]), fabsf(x[2])), m1 = fmax3(fabsf(x[3]), fabsf(x[4]), fabsf(x[5]));
  float m2 = fmax3(fabsf(x[6]), fabsf(x[7]), fabsf(x[8])), m3 = fmax3(fabsf(x[9]), fabsf(x[10]), fabsf(x[11]));
#pragma unroll
  for (int i = 12; i < 28; i += 8) {
    m0 = fmax3(m0, fabsf(x[i]), fabsf(x[i + 1]));
    m1 = fmax3(m1, fabsf(x[i + 2]), fabsf(x[i + 3]));
    m2 = fmax3(m2, fabsf(x[i + 4]), fabsf(x[i + 5]));
    m3 = fmax3(m3, fabsf(x[i + 6]), fabsf(x[i + 7]));
  }
  m0 = fmax3(m0, fabsf(x[28]), fabsf(x[29]));
  m1 = fmax3(m1, fabsf(x[30]), fabsf(x[31]));
  float am = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  am = warp_max_abs(am);
  // an all-zero block keeps the unit scale whatever its boost
  int e = am == 0.0f ? 0 : mx_exponent_bits(__float_as_uint(am)) - shift;
  if (e < -127) e = -127;
  const float sc = exp2i_neg(e + shift);
  const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 a = f2_unpack(f2_mul(f2_pack(x[4 * k], x[4 * k + 1]), sc2));
    const float2 b = f2_unpack(f2_mul(f2_pack(x[4 * k + 2], x[4 * k + 3]), sc2));
    w[k] = pack_e4m3x4(a.x, a.y, b.x, b.y);
  }
  return static_cast<uint32_t>(e + 127);
}

// Strict dQ operand: the 32 x 32 block one row per lane (x: this lane's 32
// values, columns 0..31, carrying a 2^shift boost) times f, quantized with
// one exponent per column -- from the column's max over the 32 lanes by the
// MX rule, of the values without their boost; an all-zero column keeps the
// unit scale -- into w (byte c of this lane's row).  Returns the UE8M0 byte
// of column `lane`.  The column maxima come from a transpose-reduce: at the
// step of distance o every lane keeps the half of its columns that matches
// bit o of its lane and takes the partner's maxima of that half, so after
// five steps lane c holds column c's max (31 shuffles); each lane then forms
// one exponent, and the 32 scale factors go back by shuffles.
__device__ __forceinline__ uint8_t quant_ds_cols32(const float (&x)[32], int shift, float f, int lane,
                                                   uint32_t (&w)[8]) {
  float m[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) m[c] = fabsf(x[c] * f);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = hi ? m[i] : m[i + o];
      const float keep = hi ? m[i + o] : m[i];
      m[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  // m[0] is the max of column `lane`
  int e = m[0] == 0.0f ? 0 : mx_exponent_bits(__float_as_uint(m[0])) - shift;
  if (e < -127) e = -127;
  const float sc = exp2i_neg(e + shift);
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float s0 = __shfl_sync(0xffffffffu, sc, c), s1 = __shfl_sync(0xffffffffu, sc, c + 1);
    const float s2 = __shfl_sync(0xffffffffu, sc, c + 2), s3 = __shfl_sync(0xffffffffu, sc, c + 3);
    w[c >> 2] = pack_e4m3x4(x[c] * f * s0, x[c + 1] * f * s1, x[c + 2] * f * s2, x[c + 3] * f * s3);
  }
  return static_cast<uint8_t>(e + 127);
}

}  // namespace mxa
