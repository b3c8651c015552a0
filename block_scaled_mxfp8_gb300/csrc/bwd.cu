// bwd.cu -- MXFP8 block-scaled attention backward (tcgen05, TMEM, TMA).
//
// The D prep and the key-bound passes of every backward call, and the fused
// backward of the FP16 x 2^9 dQ mode when the workspace cannot hold the
// emitted dS (the other modes and workspaces run the dK/dV kernel and a dQ
// kernel of their own).  The fused path is three launches (FLAMIA notes
// sec. 2 and Algorithm 1, steps 09-16):
//   bwd_prep_kernel   : D_i = sum_c G_ic O_ic with G from its ROW view (the
//                       same G representation the dP product uses) and O the
//                       forward's bf16 output.
//   attn_bwd_kernel   : one CTA per (128-key tile, kv head, document); loops
//                       over the query heads of the kv group and the visible
//                       128-query tiles:
//                         S^T  = K Q^T            (ROW views)
//                         P^T  = exp(alpha S^T - LSE)  (the forward's exp rule)
//                         dP^T = V G^T            (ROW views)
//                         dS^T = P^T (dP^T - D), quantized per 32 x 32 block
//                                from the block max-abs, taken with a warp
//                                max reduction in the register layout (a warp
//                                owns 32 key rows) -- no transpose (FA4
//                                write-up, "Квантование dS без транспонирования")
//                         dV  += E4M3(2^8 P^T) G  (scale 2^-8; G TOK view)
//                         dK  += dS^T Q           (Q TOK view)
//                         dQ_i = dS K             (K TOK view; the dS^T codes in
//                                shared memory read as an MN-major operand)
//                       dQ_i is added to a global fp16 accumulator after a
//                       2^9 boost (the kernel's fp32 branch is not reached
//                       from the library's entry points).
//   dq_convert_kernel : dQ = acc * 2^-9 (fp16) -> bf16.
//
// TMEM columns (512): X [0,128) holds S^T, then dP^T, then the dQ tile;
// dV [128,256), dK [256,384); P^T codes [384,416), dS^T codes [416,448);
// scale factors from 448 (4 columns each).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "attn_common.cuh"

namespace mxa {

namespace {

template <int D>
struct BwdCfg {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  static constexpr int kThreads = 256;
  // TMEM columns
  static constexpr uint32_t kColX = 0, kColDV = 128, kColDK = 256, kColP = 384, kColDS = 416;
  static constexpr uint32_t kSfK = 448, kSfQ = 452 /*+4s*/, kSfV = 460, kSfG = 464 /*+4s*/, kSfP = 472,
                            kSfGt = 476 /*+4s*/, kSfDSk = 484, kSfQt = 488 /*+4s*/, kSfDSq = 496, kSfKt = 500;
  // shared memory (offsets from the 1024-aligned base)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffKt = kOffV + kTileBytes;
  static constexpr int kOffDS = kOffKt + kTileBytes;                 // 128 x 128 dS^T codes, SW128
  static constexpr int kOffStage = kOffDS + 128 * 128;               // per-stage Q, G, Qt, Gt tiles
  static constexpr int kStageBytes = 4 * kTileBytes;
  static constexpr int kOffSf = kOffStage + kStages * kStageBytes;   // atoms: K, V, Kt, then 4 per stage
  static constexpr int kOffLse = kOffSf + (3 + 4 * kStages) * kAtomBytes;  // 2 x 128 floats
  static constexpr int kOffDv = kOffLse + 2 * 128 * 4;                      // 2 x 128 floats
  static constexpr int kSmemBytes = kOffDv + 2 * 128 * 4 + 1024;
};






}  // namespace

// ----------------------------------------------------------------- D prep
// D_i = sum_c G~row_ic O_ic and LSE_i * log2(e), written tile-padded
// [Hq, NT, 128] so that the backward kernels fetch a tile's 128 values with
// one bulk copy; rows past a document's end get D = 0 and LSE = +inf (their
// recomputed P is exp(-inf) = 0).  One CTA per (128-token tile, doc, head),
// one warp per row.
// Each warp takes its rows kRows at a time, with every load of those rows
// issued before the first sum (read-only loads, so that the D and LSE stores of the
// previous rows do not hold them back).  Per row the arithmetic is the same:
// a lane's D partial over its channels in one fixed order, then the warp sum.
template <int D>
__global__ void __launch_bounds__(256, 4) bwd_prep_kernel(PrepArgs a) {
  constexpr int kCh = D / 32;  // channels per lane
  constexpr int kRows = 8;     // rows of a warp in flight (of its 16)
  using CodeT = typename std::conditional<D == 128, uint32_t, uint16_t>::type;
  using OT = typename std::conditional<D == 128, uint2, uint32_t>::type;
  __shared__ int64_t s_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  if (static_cast<int64_t>(i) * 128 >= n) return;
  const int64_t tb = doc_tile_base(a.cu_seqlens, b, n, tid, 256, &s_slot);
  const int64_t slot = (static_cast<int64_t>(h) * a.ntiles + tb + i) * 128;
  const uint8_t* atom = a.g_sf + (static_cast<int64_t>(h) * a.ntiles + tb + i) * kAtomBytes;
  const int c0 = kCh * lane;  // this lane's first channel (all in group c0 / 32)
  const CodeT* gcodes = reinterpret_cast<const CodeT*>(a.g_codes);
  const OT* orow = reinterpret_cast<const OT*>(a.o);
#pragma unroll 1
  for (int r0 = warp; r0 < 128; r0 += 8 * kRows) {  // rows r0 + 8 q
    CodeT codes[kRows];
    OT ov[kRows];
    uint32_t sb[kRows];
    float lse[kRows];
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      const int r = r0 + 8 * q;
      const int64_t pos = static_cast<int64_t>(i) * 128 + r;
      const int64_t t = doc_start + (pos < n ? pos : 0);
      codes[q] = __ldg(gcodes + (t * a.Hq + h) * (D / kCh) + lane);
      ov[q] = __ldg(orow + (t * a.Hq + h) * (D / kCh) + lane);
      sb[q] = __ldg(atom + atom_offset(r, c0 / 32));
      lse[q] = lane == 0 ? __ldg(a.lse + static_cast<int64_t>(h) * a.T + t) : 0.0f;
    }
    float acc[kRows];
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      const float sc = exp2f(static_cast<float>(static_cast<int>(sb[q]) - 127));
      if constexpr (D == 128) {
        const float2 g01 = e4m3x2_to_f32x2(codes[q] & 0xFFFFu), g23 = e4m3x2_to_f32x2(codes[q] >> 16);
        acc[q] = (g01.x * __uint_as_float(ov[q].x << 16) + g01.y * __uint_as_float(ov[q].x & 0xFFFF0000u) +
                  g23.x * __uint_as_float(ov[q].y << 16) + g23.y * __uint_as_float(ov[q].y & 0xFFFF0000u)) * sc;
      } else {
        const float2 g01 = e4m3x2_to_f32x2(codes[q]);
        acc[q] = (g01.x * __uint_as_float(ov[q] << 16) + g01.y * __uint_as_float(ov[q] & 0xFFFF0000u)) * sc;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
      for (int q = 0; q < kRows; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
    }
#pragma unroll
    for (int q = 0; q < kRows; ++q) {
      const int r = r0 + 8 * q;
      const int64_t pos = static_cast<int64_t>(i) * 128 + r;
      if (pos >= n) {  // past the document's end: P = exp(-inf) = 0
        if (lane == 0) {
          a.dpad[slot + r] = 0.0f;
          a.lpad[slot + r] = INFINITY;
        }
        continue;
      }
      if (lane == 0) {
        a.dpad[slot + r] = acc[q];
        a.lpad[slot + r] = lse[q] * 1.4426950408889634f;
      }
      if (a.dq_boost != nullptr) {
        // g_i = cl2(max_c |G~_ic|): this lane's codes (one 32-channel group)
        // with the group's scale, then the warp maximum
        const int64_t t = doc_start + pos;
        uint32_t w = static_cast<uint32_t>(codes[q]) & 0x7F7F7F7Fu;
        w = __vmaxu4(w, w >> 16);
        w = __vmaxu4(w, w >> 8);
        const uint32_t cmax = w & 0xFFu;
        int g = cmax ? cl2_e4m3(cmax) + static_cast<int>(sb[q]) - 127 : kCl2None;
        g = __reduce_max_sync(0xffffffffu, g);
        if (lane == 0) {
          const int64_t nvis = a.causal ? pos + 1 : n;
          const int lg = cl2_count(nvis);
          const int sp = 1 + (lg > 14 ? lg - 14 : 0);
          const int kb = a.key_bound[t * a.Hkv + h / (a.Hq / a.Hkv)];
          int beta = 11 - cl2_f32(a.alpha) - (D == 128 ? 7 : 6) - sp - g - kb;
          beta = beta < -100 ? -100 : (beta > 100 ? 100 : beta);
          a.dq_boost[static_cast<int64_t>(h) * a.T + t] = __uint_as_float(static_cast<uint32_t>(beta + 127) << 23);
        }
      }
    }
  }
}

// ----------------------------------------------------------------- key bound
// FP16 per-row boost (FLAMIA notes sec. 4, the strict accumulator scale): for
// every (key token j, kv head), v_j = cl2(max_c |V~_jc|) and k_j =
// cl2(max_c |K~_jc|) from the ROW views, and the bound a query at position j
// uses: the running maxima of v and k over the document's keys up to j
// (causal), or over the whole document, summed.  Two passes over 128-token
// tiles: per-token values and tile maxima, then the prefix over the tiles.
namespace {

// cl2(max_c |x~_c|) of one ROW-view vector of D codes (D / 32 groups of 32
// codes with their scale bytes), or kCl2None; the codes are already loaded.
template <int D>
__device__ __forceinline__ int row_cl2max(const uint4 (&w)[D / 16], const uint8_t* atom, int r) {
  int best = kCl2None;
#pragma unroll
  for (int g = 0; g < D / 32; ++g) {
    const uint4 x = w[2 * g], y = w[2 * g + 1];
    uint32_t m = __vmaxu4(__vmaxu4(__vmaxu4(x.x & 0x7F7F7F7Fu, x.y & 0x7F7F7F7Fu),
                                   __vmaxu4(x.z & 0x7F7F7F7Fu, x.w & 0x7F7F7F7Fu)),
                          __vmaxu4(__vmaxu4(y.x & 0x7F7F7F7Fu, y.y & 0x7F7F7F7Fu),
                                   __vmaxu4(y.z & 0x7F7F7F7Fu, y.w & 0x7F7F7F7Fu)));
    m = __vmaxu4(m, m >> 16);
    m = __vmaxu4(m, m >> 8);
    const uint32_t c = m & 0xFFu;
    if (c) {
      const int e = cl2_e4m3(c) + static_cast<int>(atom[atom_offset(r, g)]) - 127;
      best = e > best ? e : best;
    }
  }
  return best;
}

}  // namespace

__device__ __forceinline__ uint32_t pack_vk(int v, int k) {
  return (static_cast<uint32_t>(v & 0xFFFF) << 16) | static_cast<uint32_t>(k & 0xFFFF);
}
__device__ __forceinline__ int unpack_v(uint32_t x) { return static_cast<int16_t>(x >> 16); }
__device__ __forceinline__ int unpack_k(uint32_t x) { return static_cast<int16_t>(x & 0xFFFFu); }

// Pass 1, one CTA per (128-token tile, document, kv head), one thread per
// token: v_j and k_j (int16 each, packed into key_bound) and the tile's maxima.
// Both code rows are loaded before any arithmetic (2 D bytes in flight per
// thread).
template <int D>
__global__ void __launch_bounds__(128) key_bound_tiles_kernel(KeyBoundArgs a) {
  __shared__ int s_m[2][4];
  __shared__ int64_t s_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, b = blockIdx.y, hk = blockIdx.z;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  if (static_cast<int64_t>(tile) * 128 >= n) return;
  const int64_t tb = doc_tile_base(a.cu_seqlens, b, n, tid, 128, &s_slot);
  const int64_t pos = static_cast<int64_t>(tile) * 128 + tid;
  int v = kCl2None, k = kCl2None;
  if (pos < n) {
    const int64_t t = doc_start + pos;
    const int64_t atom = (static_cast<int64_t>(hk) * a.ntiles + tb + tile) * kAtomBytes;
    uint4 wv[D / 16], wk[D / 16];
    const uint4* pv = reinterpret_cast<const uint4*>(a.v_codes + (t * a.Hkv + hk) * D);
    const uint4* pk = reinterpret_cast<const uint4*>(a.k_codes + (t * a.Hkv + hk) * D);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      wv[i] = __ldg(pv + i);
      wk[i] = __ldg(pk + i);
    }
    v = row_cl2max<D>(wv, a.v_sf + atom, tid);
    k = row_cl2max<D>(wk, a.k_sf + atom, tid);
    a.key_bound[t * a.Hkv + hk] = static_cast<int32_t>(pack_vk(v, k));
  }
  v = __reduce_max_sync(0xffffffffu, v);
  k = __reduce_max_sync(0xffffffffu, k);
  if (lane == 0) {
    s_m[0][warp] = v;
    s_m[1][warp] = k;
  }
  __syncthreads();
  if (tid == 0) {
    const int vm = max(max(s_m[0][0], s_m[0][1]), max(s_m[0][2], s_m[0][3]));
    const int km = max(max(s_m[1][0], s_m[1][1]), max(s_m[1][2], s_m[1][3]));
    a.tile_max[static_cast<int64_t>(hk) * a.ntiles + tb + tile] = static_cast<int32_t>(pack_vk(vm, km));
  }
}

// Pass 2, same grid: the maxima of the earlier tiles of the document (causal)
// or of all its tiles, then the running maxima inside the tile (causal), and
// key_bound = V + K.
__global__ void __launch_bounds__(128) key_bound_scan_kernel(KeyBoundArgs a) {
  __shared__ int s_m[2][4];
  __shared__ int64_t s_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, b = blockIdx.y, hk = blockIdx.z;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  if (static_cast<int64_t>(tile) * 128 >= n) return;
  const int64_t tb = doc_tile_base(a.cu_seqlens, b, n, tid, 128, &s_slot);
  const int ntl = static_cast<int>((n + 127) / 128);
  const int upto = a.causal ? tile : ntl;
  int cv = kCl2None, ck = kCl2None;
  for (int i = tid; i < upto; i += 128) {
    const uint32_t x = static_cast<uint32_t>(a.tile_max[static_cast<int64_t>(hk) * a.ntiles + tb + i]);
    cv = max(cv, unpack_v(x));
    ck = max(ck, unpack_k(x));
  }
  cv = __reduce_max_sync(0xffffffffu, cv);
  ck = __reduce_max_sync(0xffffffffu, ck);
  if (lane == 0) {
    s_m[0][warp] = cv;
    s_m[1][warp] = ck;
  }
  __syncthreads();
  cv = max(max(s_m[0][0], s_m[0][1]), max(s_m[0][2], s_m[0][3]));
  ck = max(max(s_m[1][0], s_m[1][1]), max(s_m[1][2], s_m[1][3]));
  const int64_t pos = static_cast<int64_t>(tile) * 128 + tid;
  const int64_t t = doc_start + pos;
  if (!a.causal) {
    if (pos < n) a.key_bound[t * a.Hkv + hk] = cv + ck;
    return;
  }
  int v = kCl2None, k = kCl2None;
  if (pos < n) {
    const uint32_t x = static_cast<uint32_t>(a.key_bound[t * a.Hkv + hk]);
    v = unpack_v(x);
    k = unpack_k(x);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yv = __shfl_up_sync(0xffffffffu, v, o), yk = __shfl_up_sync(0xffffffffu, k, o);
    if (lane >= o) {
      v = max(v, yv);
      k = max(k, yk);
    }
  }
  __syncthreads();  // the carry has been read from s_m
  if (lane == 31) {
    s_m[0][warp] = v;
    s_m[1][warp] = k;
  }
  __syncthreads();
  for (int w = 0; w < warp; ++w) {
    v = max(v, s_m[0][w]);
    k = max(k, s_m[1][w]);
  }
  if (pos < n) a.key_bound[t * a.Hkv + hk] = max(v, cv) + max(k, ck);
}

// ----------------------------------------------------------------- dQ convert
__global__ void __launch_bounds__(256) dq_convert_kernel(DqConvArgs a) {
  const int64_t n4 = a.n / 4;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.dq);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v0, v1, v2, v3;
    if (a.mode == 0) {
      const float4 f = reinterpret_cast<const float4*>(a.acc32)[i];
      v0 = f.x, v1 = f.y, v2 = f.z, v3 = f.w;
    } else {
      const uint2 hv = reinterpret_cast<const uint2*>(a.acc16)[i];
      const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
      const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
      const float inv = 1.0f / 512.0f;
      v0 = f01.x * inv, v1 = f01.y * inv, v2 = f23.x * inv, v3 = f23.y * inv;
    }
    __nv_bfloat162 b0 = __floats2bfloat162_rn(v0, v1), b1 = __floats2bfloat162_rn(v2, v3);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&b0);
    o.y = *reinterpret_cast<uint32_t*>(&b1);
    reinterpret_cast<uint2*>(out)[i] = o;
  }
}

// ----------------------------------------------------------------- main
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_kv, bar_tile_full[C::kStages], bar_tile_empty[C::kStages], bar_s_full, bar_x_free,
      bar_dp_full, bar_p_ready, bar_dq_full, bar_x_free2, bar_final, bar_drain, bar_lse[2], bar_e[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot;
  __shared__ uint32_t s_e[2][4][4];  // dS block exponent bytes [parity][key block][query block]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kt = blockIdx.x, b = blockIdx.y, hk = blockIdx.z;
  const int grp = a.Hq / a.Hkv;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  const int n_tiles = static_cast<int>((n + 127) / 128);
  if (kt >= n_tiles) return;
  const int qi0 = a.causal ? kt : 0;
  const int nq = n_tiles - qi0;       // query tiles per head
  const int n_work = nq * grp;        // (head, query tile) items
  const int64_t tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, C::kThreads, &s_slot);

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_tile_full[s], 1);
      mbar_init(&bar_tile_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_x_free, 128);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_ready, 128);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_x_free2, 128);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_lse[i], 128);
      mbar_init(&bar_e[i], 128);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sKt = smem + C::kOffKt;
  uint8_t* sDS = smem + C::kOffDS;
  uint8_t* sSf = smem + C::kOffSf;  // [0]=K, [1]=V, [2]=Kt, then stage s: 3+4s .. (Q, G, Qt, Gt)
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sDv = reinterpret_cast<float*>(smem + C::kOffDv);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.g);
      tma_prefetch_desc(&maps.qt);
      tma_prefetch_desc(&maps.gt);
      const int64_t k0 = doc_start + static_cast<int64_t>(kt) * 128;
      const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles + tile_base + kt) * kAtomBytes;
      mbar_arrive_expect_tx(&bar_kv, 3 * C::kTileBytes + 3 * kAtomBytes);
      tma_load_3d(sK, &maps.k, &bar_kv, 0, hk, static_cast<int>(k0));
      tma_load_3d(sV, &maps.v, &bar_kv, 0, hk, static_cast<int>(k0));
      tma_load_3d(sKt, &maps.kt, &bar_kv, 0, hk, static_cast<int>(k0));
      bulk_load(sSf + 0 * kAtomBytes, a.k_sf + katom, kAtomBytes, &bar_kv);
      bulk_load(sSf + 1 * kAtomBytes, a.v_sf + katom, kAtomBytes, &bar_kv);
      bulk_load(sSf + 2 * kAtomBytes, a.kt_sf + katom, kAtomBytes, &bar_kv);
      int issued = 0;
      for (int u = 0; u < n_work; ++u) {
        const int s = u % C::kStages;
        if (u >= C::kStages &&
            !role_wait(&bar_tile_empty[s], ((u / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        const int h = hk * grp + u / nq;
        const int qi = qi0 + u % nq;
        const int64_t q0 = doc_start + static_cast<int64_t>(qi) * 128;
        const int64_t qatom = (static_cast<int64_t>(h) * a.ntiles + tile_base + qi) * kAtomBytes;
        uint8_t* st = smem + C::kOffStage + s * C::kStageBytes;
        uint8_t* sf = sSf + (3 + 4 * s) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_tile_full[s], 4 * C::kTileBytes + 4 * kAtomBytes);
        tma_load_3d(st + 0 * C::kTileBytes, &maps.q, &bar_tile_full[s], 0, h, static_cast<int>(q0));
        tma_load_3d(st + 1 * C::kTileBytes, &maps.g, &bar_tile_full[s], 0, h, static_cast<int>(q0));
        tma_load_3d(st + 2 * C::kTileBytes, &maps.qt, &bar_tile_full[s], 0, h, static_cast<int>(q0));
        tma_load_3d(st + 3 * C::kTileBytes, &maps.gt, &bar_tile_full[s], 0, h, static_cast<int>(q0));
        bulk_load(sf + 0 * kAtomBytes, a.q_sf + qatom, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 1 * kAtomBytes, a.g_sf + qatom, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 2 * kAtomBytes, a.qt_sf + qatom, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 3 * kAtomBytes, a.gt_sf + qatom, kAtomBytes, &bar_tile_full[s]);
        issued = u + 1;
      }
      role_wait(&bar_kv, 0, abort_flag, nullptr, 0);
      for (int u = (issued > C::kStages ? issued - C::kStages : 0); u < issued; ++u)
        mbar_wait(&bar_tile_full[u % C::kStages], (u / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = role_wait(&bar_kv, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfK, sSf + 0 * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfV, sSf + 1 * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfKt, sSf + 2 * kAtomBytes);
      }
      const uint32_t ka = smem_u32(sK), va = smem_u32(sV), kta = smem_u32(sKt), dsa = smem_u32(sDS);
      for (int u = 0; ok && u < n_work; ++u) {
        const int s = u % C::kStages;
        const uint32_t st = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
        const uint8_t* sf = sSf + (3 + 4 * s) * kAtomBytes;
        if (!(ok = role_wait(&bar_tile_full[s], (u / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        // X must be free: the previous dQ tile has been read out
        if (u > 0 && !(ok = role_wait(&bar_x_free2, (u - 1) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        // S^T = K Q^T
        tmem_cp_atom(tmem + C::kSfQ + 4 * s, sf + 0 * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColX, make_sdesc(ka + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + 0 * C::kTileBytes + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tmem + C::kSfK, tmem + C::kSfQ + 4 * s, kk > 0);
        mma_commit(&bar_s_full);
        // dP^T = V G^T, once the softmax warps have read S^T out of X
        if (!(ok = role_wait(&bar_x_free, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfG + 4 * s, sf + 1 * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColX, make_sdesc(va + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + 1 * C::kTileBytes + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tmem + C::kSfV, tmem + C::kSfG + 4 * s, kk > 0);
        mma_commit(&bar_dp_full);
        // gradients, once P^T, dS^T and their scales are in place
        if (!(ok = role_wait(&bar_p_ready, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfGt + 4 * s, sf + 3 * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfQt + 4 * s, sf + 2 * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dV += P^T G  (contraction over 128 queries)
          mma_mxf8_ts(tmem + C::kColDV, tmem + C::kColP + 8 * kk,
                      make_sdesc(st + 3 * C::kTileBytes + kk * 32 * D, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, D, 0, 1, kk, kk), tmem + C::kSfP, tmem + C::kSfGt + 4 * s,
                      (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dK += dS^T Q
          mma_mxf8_ts(tmem + C::kColDK, tmem + C::kColDS + 8 * kk,
                      make_sdesc(st + 2 * C::kTileBytes + kk * 32 * D, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, D, 0, 1, kk, kk), tmem + C::kSfDSk, tmem + C::kSfQt + 4 * s,
                      (u > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dQ tile = dS K  (contraction over 128 keys)
          mma_mxf8_ss(tmem + C::kColX, make_sdesc(dsa + kk * 32 * 128, 16, 1024, kSwz128),
                      make_sdesc(kta + kk * 32 * D, 16, C::kSBO, C::kSwz), make_idesc_mxf8(128, D, 1, 1, kk, kk),
                      tmem + C::kSfDSq, tmem + C::kSfKt, kk > 0 ? 1u : 0u);
        mma_commit(&bar_dq_full);
        mma_commit(&bar_tile_empty[s]);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS / epilogues
    const int quad = warp & 3;
    const int j = quad * 32 + lane;  // key row of this thread (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t kpos = static_cast<int64_t>(kt) * 128 + j;
    const bool key_valid = kpos < n;
    const float sl2 = a.scale_log2;
    // constant P^T scale 2^-8
    tmem_st4(lane_base + C::kSfP, 0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
    tmem_st_wait();
    bool ok = true;
    for (int u = 0; u < n_work; ++u) {
      const int h = hk * grp + u / nq;
      const int qi = qi0 + u % nq;
      const int par = u & 1;
      // LSE (log2 units) and D of the 128 queries of this tile
      {
        const int c = quad * 32 + lane;
        const int64_t qp = static_cast<int64_t>(qi) * 128 + c;
        float l2 = 0.0f, dd = 0.0f;
        if (qp < n) {
          const int64_t slot = (static_cast<int64_t>(h) * a.ntiles + tile_base + qi) * 128 + c;
          l2 = a.lpad[slot];
          dd = a.dpad[slot];
        }
        sLse[par * 128 + c] = l2;
        sDv[par * 128 + c] = dd;
      }
      mbar_arrive(&bar_lse[par]);
      ok = role_wait(&bar_lse[par], (u >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      ok = role_wait(&bar_s_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float p[128];
      {
        uint32_t rr[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(lane_base + C::kColX + 32 * c, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) p[32 * c + i] = __uint_as_float(rr[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_x_free);
      const int64_t qbase = static_cast<int64_t>(qi) * 128;
      const bool full = key_valid && (qbase + 127 < n) && (!a.causal || kpos <= qbase);
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const float v = ex2_approx(fmaf(p[c], sl2, -sLse[par * 128 + c]));
        const int64_t qp = qbase + c;
        p[c] = (full || (key_valid && qp < n && (!a.causal || kpos <= qp))) ? v : 0.0f;
      }
      // P^T codes, boosted by 2^8 (P <= 1 after the LSE normalisation)
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w[k] = pack_e4m3x4(p[4 * (c + k)] * 256.0f, p[4 * (c + k) + 1] * 256.0f, p[4 * (c + k) + 2] * 256.0f,
                             p[4 * (c + k) + 3] * 256.0f);
        tmem_st8(lane_base + C::kColP + c, w);
      }
      ok = role_wait(&bar_dp_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t ebytes = 0;  // this warp's 4 block exponents (query block c in byte c)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColX + 32 * c, rr);
        tmem_ld_wait();
        float ds[32];
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          ds[i] = p[32 * c + i] * (__uint_as_float(rr[i]) - sDv[par * 128 + 32 * c + i]);
          am = fmaxf(am, fabsf(ds[i]));
        }
        // 32 x 32 block max-abs: this thread's 32 values, then the warp's 32 key rows
        am = warp_max_abs(am);
        const int e = mx_exponent_bits(__float_as_uint(am));
        const float sc = exp2i_neg(e);
        ebytes |= static_cast<uint32_t>(e + 127) << (8 * c);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w[k] = pack_e4m3x4(ds[4 * k] * sc, ds[4 * k + 1] * sc, ds[4 * k + 2] * sc, ds[4 * k + 3] * sc);
        tmem_st8(lane_base + C::kColDS + 8 * c, w);
        // row j of the dS^T tile in shared memory, 128B-swizzled (queries contiguous)
        uint4* row = reinterpret_cast<uint4*>(sDS + j * 128);
        row[(2 * c) ^ (j & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
        row[(2 * c + 1) ^ (j & 7)] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) s_e[par][quad][c] = (ebytes >> (8 * c)) & 0xFF;
      }
      mbar_arrive(&bar_e[par]);
      ok = role_wait(&bar_e[par], (u >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      {
        // dK operand A = dS^T: row = key, groups along queries -> column q = e[q][0..3]
        // dQ operand A = dS  : row = query, groups along keys -> column q = e[0..3][q]
        uint32_t ck[4], cq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ck[q] = s_e[par][q][0] | (s_e[par][q][1] << 8) | (s_e[par][q][2] << 16) | (s_e[par][q][3] << 24);
          cq[q] = s_e[par][0][q] | (s_e[par][1][q] << 8) | (s_e[par][2][q] << 16) | (s_e[par][3][q] << 24);
        }
        tmem_st4(lane_base + C::kSfDSk, ck[0], ck[1], ck[2], ck[3]);
        tmem_st4(lane_base + C::kSfDSq, cq[0], cq[1], cq[2], cq[3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_ready);
      // dQ tile (rows = queries) -> global accumulator
      ok = role_wait(&bar_dq_full, u & 1, abort_flag, a.err, kErrTimeoutEpilogue);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const int64_t qp = qbase + j;  // TMEM lane j is query row j of the dQ tile
        const bool qv = qp < n;
        const int64_t t = doc_start + qp;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(lane_base + C::kColX + 32 * c, rr);
          tmem_ld_wait();
          if (qv) {
            if (a.dq_mode == 0) {
              float* dst = a.dq_acc32 + (t * a.Hq + h) * D + 32 * c;
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(dst + i),
                             "f"(__uint_as_float(rr[i]) * a.alpha), "f"(__uint_as_float(rr[i + 1]) * a.alpha),
                             "f"(__uint_as_float(rr[i + 2]) * a.alpha), "f"(__uint_as_float(rr[i + 3]) * a.alpha)
                             : "memory");
            } else {
              uint16_t* dst = a.dq_acc16 + (t * a.Hq + h) * D + 32 * c;
              const float bst = a.alpha * 512.0f;
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint32_t hw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  __half2 hv = __floats2half2_rn(__uint_as_float(rr[i + 2 * k]) * bst, __uint_as_float(rr[i + 2 * k + 1]) * bst);
                  hw[k] = *reinterpret_cast<uint32_t*>(&hv);
                }
                asm volatile("red.global.add.noftz.v4.f16x2 [%0], {%1,%2,%3,%4};" ::"l"(dst + i), "r"(hw[0]),
                             "r"(hw[1]), "r"(hw[2]), "r"(hw[3])
                             : "memory");
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_x_free2);
    }
    // ---------------------------------------------------------- dK, dV out
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = doc_start + kpos;
      __nv_bfloat16* dvrow = reinterpret_cast<__nv_bfloat16*>(a.dv) + (t * a.Hkv + hk) * D;
      __nv_bfloat16* dkrow = reinterpret_cast<__nv_bfloat16*>(a.dk) + (t * a.Hkv + hk) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
        const float mul = which == 0 ? 1.0f : a.alpha;
        __nv_bfloat16* dst = which == 0 ? dvrow : dkrow;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(lane_base + col + 32 * c, rr);
          tmem_ld_wait();
          if (key_valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              __nv_bfloat162 b0 = __floats2bfloat162_rn(__uint_as_float(rr[i]) * mul, __uint_as_float(rr[i + 1]) * mul);
              __nv_bfloat162 b1 = __floats2bfloat162_rn(__uint_as_float(rr[i + 2]) * mul, __uint_as_float(rr[i + 3]) * mul);
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(rr[i + 4]) * mul, __uint_as_float(rr[i + 5]) * mul);
              __nv_bfloat162 b3 = __floats2bfloat162_rn(__uint_as_float(rr[i + 6]) * mul, __uint_as_float(rr[i + 7]) * mul);
              v.x = *reinterpret_cast<uint32_t*>(&b0);
              v.y = *reinterpret_cast<uint32_t*>(&b1);
              v.z = *reinterpret_cast<uint32_t*>(&b2);
              v.w = *reinterpret_cast<uint32_t*>(&b3);
              *reinterpret_cast<uint4*>(dst + 32 * c + i) = v;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_key_bound(const KeyBoundArgs& a, int max_seqlen, cudaStream_t stream) {
  const dim3 grid((max_seqlen + 127) / 128, a.num_docs, a.Hkv);
  if (a.d == 128) key_bound_tiles_kernel<128><<<grid, 128, 0, stream>>>(a);
  else key_bound_tiles_kernel<64><<<grid, 128, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  key_bound_scan_kernel<<<grid, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const PrepArgs& a, int max_seqlen, cudaStream_t stream) {
  if (a.dq_acc_bytes && cudaMemsetAsync(a.dq_acc, 0, a.dq_acc_bytes, stream) != cudaSuccess) return cudaGetLastError();
  dim3 grid((max_seqlen + 127) / 128, a.num_docs, a.Hq);
  if (a.d == 128) bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(a);
  else bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const DqConvArgs& a, cudaStream_t stream) {
  const int64_t n4 = a.n / 4;
  int blocks = static_cast<int>((n4 + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  dq_convert_kernel<<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  dim3 grid((max_seqlen + 127) / 128, a.num_docs, a.Hkv);
  if (d == 128) {
    using C = BwdCfg<128>;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_kernel<128><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  } else {
    using C = BwdCfg<64>;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_kernel<64><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  }
  return cudaGetLastError();
}

}  // namespace mxa
