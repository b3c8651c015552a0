// fwd.cu -- MXFP8 block-scaled attention forward (tcgen05, TMEM, TMA).
//
// One CTA computes one 128-query tile of one (document, query head):
//   S_j   = Q K_j^T         block-scaled MXFP8 MMA (kind::mxf8f6f4), K-major
//                           operands, Q/K ROW-view scales in TMEM;
//   P_j   = online softmax of alpha * S_j with a lazily updated row max
//           (rescale only when the tile max exceeds the running max by more
//           than tau = 4 in log2 units), quantized in registers as
//           E4M3(2^4 * p) (FLAMIA notes sec. 5: 2^(c+tau) <= 448 with
//           (c, tau) = (4, 4)), stored to TMEM;
//   O    += P_j V_j          block-scaled MMA with A = P from TMEM (scale
//                           2^-4), B = V MN-major with TOK-view scales;
//   L    += P_j 1            the same quantized weights against a ones tile
//                           (N = 16), so that O / L is the convex combination
//                           of the V rows with exactly the weights used;
//   O = O / L -> bf16, LSE = m + ln l with l the fp32 sum of the unquantized
//   weights (FLAMIA notes sec. 2, online softmax).
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = TMEM
// owner, warps 4..11 = softmax / correction / epilogue (two warps per query
// row quadrant, each taking half of the 128 key columns).
// S is double buffered in TMEM so that S_{j+1} = Q K_{j+1}^T runs on the
// tensor core while the softmax warps work on S_j.
//
// TMEM columns: S0 [0,128) S1 [128,256) O [256,256+D) L [384,400) Q-scale 400,
// K-scale 404+4s, V-scale 416+4s, P-scale 428, ones-scale 432, P0 [448,480),
// P1 [480,512).
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace mxa {

namespace {

template <int D>
struct FwdCfg {
  static constexpr int kStages = 3;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  static constexpr int kThreads = 384;  // 4 role warps + 8 softmax warps
  static constexpr uint32_t kColS = 0, kColO = 256, kColL = 384, kColSfQ = 400, kColSfK = 404, kColSfV = 416,
                            kColSfP = 428, kColSf1 = 432, kColP = 448;
  // shared memory map (offsets from the 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffSfQ = kOffV + kStages * kTileBytes;
  static constexpr int kOffSfK = kOffSfQ + kAtomBytes;
  static constexpr int kOffSfV = kOffSfK + kStages * kAtomBytes;
  static constexpr int kOffOnes = (kOffSfV + kStages * kAtomBytes + 1023) / 1024 * 1024;  // 16 x 128 B of E4M3 1.0
  static constexpr int kSmemBytes = kOffOnes + 16 * 128 + 1024;            // + alignment slack
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_kv_full[C::kStages], bar_kv_empty[C::kStages], bar_s_full[2], bar_s_empty[2],
      bar_p_full[2], bar_o_done, bar_drain, bar_mx[2], bar_lsum;
  __shared__ float s_mx[2][2][128];  // [tile parity][half][row] partial row maxima
  __shared__ float s_l[2][128];      // [half][row] partial row sums
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y, h = blockIdx.z;
  const int hk = h / (a.Hq / a.Hkv);
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  const int nq_tiles = static_cast<int>((n + 127) / 128);
  // heaviest query tiles first when causal
  const int qt = a.causal ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  if (qt >= nq_tiles) return;
  const int n_kt = a.causal ? qt + 1 : nq_tiles;
  const int64_t tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, C::kThreads, &s_slot);

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_s_empty[i], 256);
      mbar_init(&bar_p_full[i], 256);
      mbar_init(&bar_mx[i], 256);
    }
    mbar_init(&bar_o_done, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_lsum, 256);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  for (int i = tid; i < 16 * 128 / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kOffOnes)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sSfQ = smem + C::kOffSfQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      const int64_t q0 = doc_start + static_cast<int64_t>(qt) * 128;
      mbar_arrive_expect_tx(&bar_q, C::kTileBytes + kAtomBytes);
      tma_load_3d(sQ, &maps.q, &bar_q, 0, h, static_cast<int>(q0));
      bulk_load(sSfQ, a.q_sf + ((static_cast<int64_t>(h) * a.ntiles + tile_base + qt) * kAtomBytes), kAtomBytes,
                &bar_q);
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages) {
          if (!role_wait(&bar_kv_empty[s], ((j / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma)) break;
        }
        const int64_t k0 = doc_start + static_cast<int64_t>(j) * 128;
        const int64_t atom = (static_cast<int64_t>(hk) * a.ntiles + tile_base + j) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_kv_full[s], 2 * C::kTileBytes + 2 * kAtomBytes);
        tma_load_3d(smem + C::kOffK + s * C::kTileBytes, &maps.k, &bar_kv_full[s], 0, hk, static_cast<int>(k0));
        tma_load_3d(smem + C::kOffV + s * C::kTileBytes, &maps.v, &bar_kv_full[s], 0, hk, static_cast<int>(k0));
        bulk_load(smem + C::kOffSfK + s * kAtomBytes, a.k_sf + atom, kAtomBytes, &bar_kv_full[s]);
        bulk_load(smem + C::kOffSfV + s * kAtomBytes, a.v_sf + atom, kAtomBytes, &bar_kv_full[s]);
        issued = j + 1;
      }
      // drain: every load issued must have landed before the CTA exits
      role_wait(&bar_q, 0, abort_flag, nullptr, 0);
      for (int j = (issued > C::kStages ? issued - C::kStages : 0); j < issued; ++j)
        mbar_wait(&bar_kv_full[j % C::kStages], (j / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s[4] = {make_idesc_mxf8(128, 128, 0, 0, 0, 0), make_idesc_mxf8(128, 128, 0, 0, 1, 1),
                                   make_idesc_mxf8(128, 128, 0, 0, 2, 2), make_idesc_mxf8(128, 128, 0, 0, 3, 3)};
      const uint32_t idesc_pv[4] = {make_idesc_mxf8(128, D, 0, 1, 0, 0), make_idesc_mxf8(128, D, 0, 1, 1, 1),
                                    make_idesc_mxf8(128, D, 0, 1, 2, 2), make_idesc_mxf8(128, D, 0, 1, 3, 3)};
      const uint32_t idesc_l[4] = {make_idesc_mxf8(128, 16, 0, 0, 0, 0), make_idesc_mxf8(128, 16, 0, 0, 1, 1),
                                   make_idesc_mxf8(128, 16, 0, 0, 2, 2), make_idesc_mxf8(128, 16, 0, 0, 3, 3)};
      bool ok = role_wait(&bar_q, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_atom(tmem + C::kColSfQ, sSfQ);
      }
      auto issue_s = [&](int j) -> bool {
        const int s = j % C::kStages, bb = j & 1;
        if (!role_wait(&bar_kv_full[s], (j / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        if (j >= 2 && !role_wait(&bar_s_empty[bb], ((j >> 1) - 1) & 1, abort_flag, a.err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kColSfK + 4 * s, smem + C::kOffSfK + s * kAtomBytes);
        const uint32_t qa = smem_u32(sQ), ka = smem_u32(smem + C::kOffK + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          mma_mxf8_ss(tmem + C::kColS + 128 * bb, make_sdesc(qa + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(ka + 32 * kk, 16, C::kSBO, C::kSwz), idesc_s[kk], tmem + C::kColSfQ,
                      tmem + C::kColSfK + 4 * s, kk > 0);
        }
        mma_commit(&bar_s_full[bb]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n_kt; ++j) {
        if (j + 1 < n_kt && !issue_s(j + 1)) break;
        const int s = j % C::kStages, bb = j & 1;
        if (!role_wait(&bar_p_full[bb], (j >> 1) & 1, abort_flag, a.err, kErrTimeoutMma)) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kColSfV + 4 * s, smem + C::kOffSfV + s * kAtomBytes);
        const uint32_t va = smem_u32(smem + C::kOffV + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          mma_mxf8_ts(tmem + C::kColO, tmem + C::kColP + 32 * bb + 8 * kk,
                      make_sdesc(va + kk * 32 * D, 16, C::kSBO, C::kSwz), idesc_pv[kk], tmem + C::kColSfP,
                      tmem + C::kColSfV + 4 * s, (j > 0 || kk > 0) ? 1u : 0u);
        }
        const uint32_t onesa = smem_u32(smem + C::kOffOnes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          mma_mxf8_ts(tmem + C::kColL, tmem + C::kColP + 32 * bb + 8 * kk, make_sdesc(onesa + 32 * kk, 16, 1024, kSwz128),
                      idesc_l[kk], tmem + C::kColSfP, tmem + C::kColSf1, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_o_done);
        mma_commit(&bar_kv_empty[s]);
      }
      // drain the tensor pipe before the TMEM is released
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // Two warps per TMEM lane quadrant: warp half hf handles key columns
    // [64 hf, 64 hf + 64) of its 32 rows; the halves exchange their row maxima
    // through shared memory once per tile and keep separate partial sums.
    const int quad = warp & 3;
    const int hf = (warp - 4) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t qpos = static_cast<int64_t>(qt) * 128 + r;  // document-relative query index
    const float sl2 = a.scale_log2;
    if (hf == 0) {
      // P scale 2^-4 and the ones tile's scale 1 in every cell of their columns
      tmem_st4(lane_base + C::kColSfP, 0x7B7B7B7Bu, 0x7B7B7B7Bu, 0x7B7B7B7Bu, 0x7B7B7B7Bu);
      tmem_st4(lane_base + C::kColSf1, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    float m = -INFINITY;  // running (lazy) max of the scaled scores, log2 units
    float l16 = 0.0f;     // this half's sum of 2^(s - m + 4)
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int bb = j & 1;
      if (!(ok = warp_wait(&bar_s_full[bb], (j >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      float sv[64];
      {
        uint32_t x0[32], x1[32];
        tmem_ld32(lane_base + C::kColS + 128 * bb + 64 * hf, x0);
        tmem_ld32(lane_base + C::kColS + 128 * bb + 64 * hf + 32, x1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(x0[i]);
          sv[32 + i] = __uint_as_float(x1[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_s_empty[bb]);
      if (j == n_kt - 1) {
        // keys past the document end, or (causal diagonal) after the query
        const int64_t rem = n - static_cast<int64_t>(j) * 128;
        int lim = rem < 128 ? static_cast<int>(rem) : 128;
        if (a.causal) lim = min(lim, r + 1);
        if (lim < 128) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sv[c] = (64 * hf + c < lim) ? sv[c] : -INFINITY;
        }
      }
      float mt = sv[0];
#pragma unroll
      for (int c = 1; c < 64; ++c) mt = fmaxf(mt, sv[c]);
      s_mx[bb][hf][r] = mt;
      mbar_arrive(&bar_mx[bb]);
      if (!(ok = warp_wait(&bar_mx[bb], (j >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      mt = fmaxf(mt, s_mx[bb][hf ^ 1][r]);
      const float mts = mt * sl2;
      bool rescale_o = false;
      float factor = 1.0f;
      if (j == 0) {
        m = mts;
      } else if (mts > m + 4.0f) {
        factor = ex2_approx(m - mts);
        m = mts;
        rescale_o = true;
      }
      const float neg = 4.0f - m;
      uint32_t pw[16];
      float lsum = 0.0f;
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float p0 = ex2_approx(fmaf(sv[c], sl2, neg));
        const float p1 = ex2_approx(fmaf(sv[c + 1], sl2, neg));
        const float p2 = ex2_approx(fmaf(sv[c + 2], sl2, neg));
        const float p3 = ex2_approx(fmaf(sv[c + 3], sl2, neg));
        lsum += (p0 + p1) + (p2 + p3);
        pw[c >> 2] = pack_e4m3x4(p0, p1, p2, p3);
      }
      l16 = l16 * factor + lsum;
      // tcgen05.ld/st are warp-collective: the whole warp rescales its rows'
      // half of O when any of them needs it (factor 1 for the others).
      if (__any_sync(0xffffffffu, rescale_o)) {
        if (!(ok = warp_wait(&bar_o_done, (j - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t col = C::kColO + (D / 2) * hf + 32 * c;
          uint32_t rr[32];
          tmem_ld32(lane_base + col, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(rr[i + k]) * factor);
            tmem_st8(lane_base + col + i, w);
          }
        }
        if (hf == 0) {
          uint32_t rr[16];
          tmem_ld16(lane_base + C::kColL, rr);
          tmem_ld_wait();
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(rr[k]) * factor);
          tmem_st8(lane_base + C::kColL, w);
        }
      }
#pragma unroll
      for (int c = 0; c < 16; c += 8) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = pw[c + k];
        tmem_st8(lane_base + C::kColP + 32 * bb + 16 * hf + c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p_full[bb]);
    }
    // ---------------------------------------------------------- epilogue
    s_l[hf][r] = l16;
    mbar_arrive(&bar_lsum);
    if (ok) ok = role_wait(&bar_lsum, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (ok) ok = role_wait(&bar_o_done, (n_kt - 1) & 1, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      float inv;
      {
        uint32_t rr[16];
        tmem_ld16(lane_base + C::kColL, rr);
        tmem_ld_wait();
        inv = 1.0f / __uint_as_float(rr[0]);
      }
      const bool valid = qpos < n;
      const int64_t t = doc_start + qpos;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (t * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int cb = (D / 2) * hf + 32 * c;
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColO + cb, rr);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(rr[i]) * inv, __uint_as_float(rr[i + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * inv, __uint_as_float(rr[i + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * inv, __uint_as_float(rr[i + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * inv, __uint_as_float(rr[i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cb + i) = v;
          }
        }
      }
      if (valid && hf == 0)
        a.lse[static_cast<int64_t>(h) * a.T + t] = (m - 4.0f + log2f(s_l[0][r] + s_l[1][r])) * 0.69314718055994531f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  dim3 grid((max_seqlen + 127) / 128, a.num_docs, a.Hq);
  if (d == 128) {
    using C = FwdCfg<128>;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_fwd_kernel<128><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  } else {
    using C = FwdCfg<64>;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_fwd_kernel<64><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  }
  return cudaGetLastError();
}

}  // namespace mxa
