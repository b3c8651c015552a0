// bwd_split.cu -- deterministic MXFP8 attention backward in two kernels
// (the FP32 dQ mode): no atomics, every sum in a fixed order.
//
//   attn_bwd_dkdv_kernel : one CTA per (128-key tile, kv head, document),
//       looping over the query heads of the kv group and the visible query
//       tiles (FLAMIA notes Algorithm 1 steps 11-15 without dQ):
//         S^T = K Q^T, P^T = exp(alpha S^T - LSE), dP^T = V G^T,
//         dS^T = P^T (dP^T - D) quantized per 32 x 32 block (warp max-abs in
//         the register layout: a warp holds 32 key rows, a 32-column chunk is
//         one block; no transpose),
//         dV += E4M3(2^8 P^T) G, dK += dS^T Q, both accumulated in TMEM.
//   attn_bwd_dq_kernel   : one CTA per (128-query tile, query head,
//       document), looping over the visible key tiles:
//         S = Q K^T, P = exp(alpha S - LSE), dP = G V^T,
//         dS = P (dP - D) quantized per 32 x 32 block (a warp holds 32 query
//         rows), dQ += dS K accumulated in TMEM, written once as bf16.
// Both recompute S and dP (the FLOP convention counts the backward as 2.5
// forwards; these two kernels execute 3.5).  The 32 x 32 blocks are the same
// in both kernels; each quantizes its own fp32 dS.
//
// Warps: 0 = TMA producer, 1 = MMA issuer, 2 = TMEM owner, 4..11 = softmax.
// Two softmax warps share each TMEM lane quadrant and split the tile's 128
// columns into halves of 64 (two 32 x 32 dS blocks each), so every SM
// sub-partition has two softmax warps to interleave.  The halves write their
// dS block exponents into separate scale-factor columns; the gradient MMA
// reads K steps 0-1 from the first and 2-3 from the second.
// LSE (times log2 e; +inf past a document's end) and D come tile-padded from
// the prep kernel and are bulk-loaded with the tiles.
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace mxa {

namespace {

constexpr int kSplitThreads = 384;
constexpr int kSoftmaxThreads = 256;

template <int D>
struct DkdvCfg {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  // TMEM: X holds S^T then dP^T; dV, dK accumulators; P^T and dS^T codes
  static constexpr uint32_t kColX = 0, kColDV = 128, kColDK = 256, kColP = 384, kColDS = 416;
  static constexpr uint32_t kSfK = 448, kSfQ = 452 /*+4s*/, kSfV = 460, kSfG = 464 /*+4s*/, kSfP = 472,
                            kSfGt = 476 /*+4s*/, kSfDS0 = 484, kSfDS1 = 488, kSfQt = 492 /*+4s*/;
  // shared memory: K, V, then per stage Q, G, Qt, Gt tiles + LSE + D rows
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffStage = kOffV + kTileBytes;
  static constexpr int kStageBytes = 4 * kTileBytes + 2 * 512;
  static constexpr int kOffSf = kOffStage + kStages * kStageBytes;  // K, V, then 4 per stage
  static constexpr int kSmemBytes = kOffSf + (2 + 4 * kStages) * kAtomBytes + 1024;
};

template <int D>
struct DqCfg {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  // TMEM: S and dP side by side (both MMAs issue back to back), dQ
  // accumulator, dS codes, scale atoms
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
  static constexpr uint32_t kSfQ = 416, kSfG = 420, kSfK = 424 /*+4s*/, kSfV = 432 /*+4s*/, kSfDS0 = 440,
                            kSfDS1 = 444, kSfKt = 448 /*+4s*/;
  static constexpr int kOffQ = 0;
  static constexpr int kOffG = kOffQ + kTileBytes;
  static constexpr int kOffStage = kOffG + kTileBytes;  // per stage: K, V, Kt
  static constexpr int kStageBytes = 3 * kTileBytes;
  static constexpr int kOffSf = kOffStage + kStages * kStageBytes;  // Q, G, then 3 per stage
  static constexpr int kSmemBytes = kOffSf + (2 + 3 * kStages) * kAtomBytes + 1024;
};

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&rr)[32], float mul) {
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(rr[i]) * mul, __uint_as_float(rr[i + 1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * mul, __uint_as_float(rr[i + 3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * mul, __uint_as_float(rr[i + 5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * mul, __uint_as_float(rr[i + 7]) * mul);
    *reinterpret_cast<uint4*>(dst + i) = v;
  }
}

// 64 fp32 columns of this thread's TMEM lane: two 32-column loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(a[i]);
    v[32 + i] = __uint_as_float(b[i]);
  }
}

}  // namespace

// ========================================================================= dK, dV
template <int D>
__global__ void __launch_bounds__(kSplitThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_kv, bar_tile_full[C::kStages], bar_tile_empty[C::kStages], bar_s_full, bar_x_free,
      bar_dp_full, bar_x_free2, bar_p_ready, bar_ds_ready, bar_pv_free, bar_dk_free, bar_final, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kt = blockIdx.x, b = blockIdx.y, hk = blockIdx.z;
  const int grp = a.Hq / a.Hkv;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  const int n_tiles = static_cast<int>((n + 127) / 128);
  if (kt >= n_tiles) return;
  const int qi0 = a.causal ? kt : 0;
  const int nq = n_tiles - qi0;
  const int n_work = nq * grp;
  const int64_t tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, kSplitThreads, &s_slot);

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_tile_full[s], 1);
      mbar_init(&bar_tile_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_x_free, kSoftmaxThreads);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_x_free2, kSoftmaxThreads);
    mbar_init(&bar_p_ready, kSoftmaxThreads);
    mbar_init(&bar_ds_ready, kSoftmaxThreads);
    mbar_init(&bar_pv_free, 1);
    mbar_init(&bar_dk_free, 1);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
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
  uint8_t* sSf = smem + C::kOffSf;  // [0] K, [1] V, stage s: 2 + 4s + (0 Q, 1 G, 2 Qt, 3 Gt)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const int64_t k0 = doc_start + static_cast<int64_t>(kt) * 128;
      const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles + tile_base + kt) * kAtomBytes;
      mbar_arrive_expect_tx(&bar_kv, 2 * C::kTileBytes + 2 * kAtomBytes);
      tma_load_3d(smem + C::kOffK, &maps.k, &bar_kv, 0, hk, static_cast<int>(k0));
      tma_load_3d(smem + C::kOffV, &maps.v, &bar_kv, 0, hk, static_cast<int>(k0));
      bulk_load(sSf + 0 * kAtomBytes, a.k_sf + katom, kAtomBytes, &bar_kv);
      bulk_load(sSf + 1 * kAtomBytes, a.v_sf + katom, kAtomBytes, &bar_kv);
      int issued = 0;
      for (int u = 0; u < n_work; ++u) {
        const int s = u % C::kStages;
        if (u >= C::kStages &&
            !role_wait(&bar_tile_empty[s], ((u / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        const int h = hk * grp + u / nq;
        const int qi = qi0 + u % nq;
        const int q0 = static_cast<int>(doc_start + static_cast<int64_t>(qi) * 128);
        const int64_t qslot = static_cast<int64_t>(h) * a.ntiles + tile_base + qi;
        uint8_t* st = smem + C::kOffStage + s * C::kStageBytes;
        uint8_t* sf = sSf + (2 + 4 * s) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_tile_full[s], 4 * C::kTileBytes + 4 * kAtomBytes + 2 * 512);
        tma_load_3d(st + 0 * C::kTileBytes, &maps.q, &bar_tile_full[s], 0, h, q0);
        tma_load_3d(st + 1 * C::kTileBytes, &maps.g, &bar_tile_full[s], 0, h, q0);
        tma_load_3d(st + 2 * C::kTileBytes, &maps.qt, &bar_tile_full[s], 0, h, q0);
        tma_load_3d(st + 3 * C::kTileBytes, &maps.gt, &bar_tile_full[s], 0, h, q0);
        bulk_load(st + 4 * C::kTileBytes, a.lpad + qslot * 128, 512, &bar_tile_full[s]);
        bulk_load(st + 4 * C::kTileBytes + 512, a.dpad + qslot * 128, 512, &bar_tile_full[s]);
        bulk_load(sf + 0 * kAtomBytes, a.q_sf + qslot * kAtomBytes, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 1 * kAtomBytes, a.g_sf + qslot * kAtomBytes, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 2 * kAtomBytes, a.qt_sf + qslot * kAtomBytes, kAtomBytes, &bar_tile_full[s]);
        bulk_load(sf + 3 * kAtomBytes, a.gt_sf + qslot * kAtomBytes, kAtomBytes, &bar_tile_full[s]);
        issued = u + 1;
      }
      role_wait(&bar_kv, 0, abort_flag, nullptr, 0);
      for (int u = (issued > C::kStages ? issued - C::kStages : 0); u < issued; ++u)
        mbar_wait(&bar_tile_full[u % C::kStages], (u / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t ka = smem_u32(smem + C::kOffK), va = smem_u32(smem + C::kOffV);
      bool ok = role_wait(&bar_kv, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfK, sSf + 0 * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfV, sSf + 1 * kAtomBytes);
      }
      auto issue_s = [&](int u) -> bool {  // S^T = K Q^T into X
        const int s = u % C::kStages;
        if (!role_wait(&bar_tile_full[s], (u / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
        tmem_cp_atom(tmem + C::kSfQ + 4 * s, sSf + (2 + 4 * s + 0) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColX, make_sdesc(ka + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + 32 * kk, 16, C::kSBO, C::kSwz), make_idesc_mxf8(128, 128, 0, 0, kk, kk),
                      tmem + C::kSfK, tmem + C::kSfQ + 4 * s, kk > 0);
        mma_commit(&bar_s_full);
        return true;
      };
      // Pipe order per unit u: dP^T_u, dV_u, S^T_{u+1}, dK_u.  X is written
      // only by S^T and dP^T; between two writes of X the pipe always holds
      // an MMA that does not touch X (dV_u, dK_u), which covers the softmax
      // warps' read of X.
      if (ok) ok = issue_s(0);
      for (int u = 0; ok && u < n_work; ++u) {
        const int s = u % C::kStages;
        const uint32_t st = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
        // dP^T = V G^T once S^T has been read out of X
        if (!(ok = role_wait(&bar_x_free, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfG + 4 * s, sSf + (2 + 4 * s + 1) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColX, make_sdesc(va + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + C::kTileBytes + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tmem + C::kSfV, tmem + C::kSfG + 4 * s, kk > 0);
        mma_commit(&bar_dp_full);
        // dV += P^T G (P^T codes written while dP^T ran)
        if (!(ok = role_wait(&bar_p_ready, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfGt + 4 * s, sSf + (2 + 4 * s + 3) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf8_ts(tmem + C::kColDV, tmem + C::kColP + 8 * kk,
                      make_sdesc(st + 3 * C::kTileBytes + kk * 32 * D, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, D, 0, 1, kk, kk), tmem + C::kSfP, tmem + C::kSfGt + 4 * s,
                      (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_pv_free);
        // next S^T as soon as dP^T has been read (runs while dS is formed)
        if (!(ok = role_wait(&bar_x_free2, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (u + 1 < n_work && !(ok = issue_s(u + 1))) break;
        // dK += dS^T Q
        if (!(ok = role_wait(&bar_ds_ready, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfQt + 4 * s, sSf + (2 + 4 * s + 2) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf8_ts(tmem + C::kColDK, tmem + C::kColDS + 8 * kk,
                      make_sdesc(st + 2 * C::kTileBytes + kk * 32 * D, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, D, 0, 1, kk & 1, kk), tmem + (kk < 2 ? C::kSfDS0 : C::kSfDS1),
                      tmem + C::kSfQt + 4 * s, (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_dk_free);
        mma_commit(&bar_tile_empty[s]);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    const int quad = warp & 3;
    const int hf = (warp - 4) >> 2;       // column half: queries [64 hf, 64 hf + 64)
    const int j = quad * 32 + lane;       // key row (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t kpos = static_cast<int64_t>(kt) * 128 + j;
    const bool key_valid = kpos < n;
    const float kb8 = key_valid ? 8.0f : -INFINITY;  // 2^8 boost of P^T; invalid key rows -> 0
    const float sl2 = a.scale_log2;
    if (hf == 0) {
      tmem_st4(lane_base + C::kSfP, 0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);  // 2^-8
      tmem_st_wait();
    }
    bool ok = true;
    for (int u = 0; u < n_work; ++u) {
      const int s = u % C::kStages;
      const int qi = qi0 + u % nq;
      const float* lrow = reinterpret_cast<const float*>(smem + C::kOffStage + s * C::kStageBytes + 4 * C::kTileBytes) + 64 * hf;
      const float* drow = lrow + 128;
      if (!(ok = warp_wait(&bar_s_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      float p[64];
      tmem_ld64(lane_base + C::kColX + 64 * hf, p);
      tc_fence_before();
      mbar_arrive(&bar_x_free);
      // P^T boosted by 2^8 (P <= 1 after the LSE normalization); rows past the
      // document end have LSE = +inf, so their P is 0 without a test
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lrow + c);
        p[c] = ex2_approx(fmaf(p[c], sl2, kb8 - l4.x));
        p[c + 1] = ex2_approx(fmaf(p[c + 1], sl2, kb8 - l4.y));
        p[c + 2] = ex2_approx(fmaf(p[c + 2], sl2, kb8 - l4.z));
        p[c + 3] = ex2_approx(fmaf(p[c + 3], sl2, kb8 - l4.w));
      }
      if (a.causal && qi == kt) {  // diagonal tile: query index (in tile) >= key index
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = (64 * hf + c >= j) ? p[c] : 0.0f;
      }
      // the previous unit's dV MMA must be done with the P^T codes
      if (u > 0 && !(ok = warp_wait(&bar_pv_free, (u - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 16; c += 8) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w[k] = pack_e4m3x4(p[4 * (c + k)], p[4 * (c + k) + 1], p[4 * (c + k) + 2], p[4 * (c + k) + 3]);
        tmem_st8(lane_base + C::kColP + 16 * hf + c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p_ready);
      if (!(ok = warp_wait(&bar_dp_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      // dS^T = P^T (dP^T - D), in place; X is released once both chunks are in
      // registers
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColX + 64 * hf + 32 * cc, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(drow + 32 * cc + i);
          p[32 * cc + i] *= __uint_as_float(rr[i]) - d4.x;
          p[32 * cc + i + 1] *= __uint_as_float(rr[i + 1]) - d4.y;
          p[32 * cc + i + 2] *= __uint_as_float(rr[i + 2]) - d4.z;
          p[32 * cc + i + 3] *= __uint_as_float(rr[i + 3]) - d4.w;
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_x_free2);
      // the previous unit's dK MMA must be done with the dS^T codes and scales
      if (u > 0 && !(ok = warp_wait(&bar_dk_free, (u - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      uint32_t ebytes = 0;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = p[32 * cc + i];
        uint32_t w[8];
        ebytes |= quant_ds_block32(x, 8, w) << (8 * cc);  // 32 key rows x 32 queries
        tmem_st8(lane_base + C::kColDS + 16 * hf + 8 * cc, w);
      }
      // dK's A operand is dS^T (rows = keys, groups = 32-query blocks); row r's
      // scales sit in lane r, column base + r / 32.  Half hf owns query
      // blocks 2 hf, 2 hf + 1 (bytes 0, 1 of its own scale columns).
      tmem_st1(lane_base + (hf ? C::kSfDS1 : C::kSfDS0) + quad, ebytes | 0x7F7F0000u);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
    }
    // ---------------------------------------------------------- dK, dV out
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = doc_start + kpos;
      __nv_bfloat16* dvrow = reinterpret_cast<__nv_bfloat16*>(a.dv) + (t * a.Hkv + hk) * D;
      __nv_bfloat16* dkrow = reinterpret_cast<__nv_bfloat16*>(a.dk) + (t * a.Hkv + hk) * D;
      // half 0 writes dV, half 1 writes dK
      const uint32_t col = hf ? C::kColDK : C::kColDV;
      __nv_bfloat16* dst = hf ? dkrow : dvrow;
      const float mul = hf ? a.alpha : 1.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + col + 32 * c, rr);
        tmem_ld_wait();
        if (key_valid) store_row_bf16(dst + 32 * c, rr, mul);
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

// ========================================================================= dQ
template <int D>
__global__ void __launch_bounds__(kSplitThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_kv_full[C::kStages], bar_kv_empty[C::kStages], bar_sdp_full, bar_x_free,
      bar_ds_ready, bar_ds_free, bar_final, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y, h = blockIdx.z;
  const int hk = h / (a.Hq / a.Hkv);
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  const int n_tiles = static_cast<int>((n + 127) / 128);
  const int qt = a.causal ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  if (qt >= n_tiles) return;
  const int n_kt = a.causal ? qt + 1 : n_tiles;
  const int64_t tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, kSplitThreads, &s_slot);

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_x_free, kSoftmaxThreads);
    mbar_init(&bar_ds_ready, kSoftmaxThreads);
    mbar_init(&bar_ds_free, 1);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
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
  uint8_t* sSf = smem + C::kOffSf;  // [0] Q, [1] G, stage s: 2 + 3s + (0 K, 1 V, 2 Kt)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const int q0 = static_cast<int>(doc_start + static_cast<int64_t>(qt) * 128);
      const int64_t qatom = (static_cast<int64_t>(h) * a.ntiles + tile_base + qt) * kAtomBytes;
      mbar_arrive_expect_tx(&bar_q, 2 * C::kTileBytes + 2 * kAtomBytes);
      tma_load_3d(smem + C::kOffQ, &maps.q, &bar_q, 0, h, q0);
      tma_load_3d(smem + C::kOffG, &maps.g, &bar_q, 0, h, q0);
      bulk_load(sSf + 0 * kAtomBytes, a.q_sf + qatom, kAtomBytes, &bar_q);
      bulk_load(sSf + 1 * kAtomBytes, a.g_sf + qatom, kAtomBytes, &bar_q);
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages &&
            !role_wait(&bar_kv_empty[s], ((j / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        const int k0 = static_cast<int>(doc_start + static_cast<int64_t>(j) * 128);
        const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles + tile_base + j) * kAtomBytes;
        uint8_t* st = smem + C::kOffStage + s * C::kStageBytes;
        uint8_t* sf = sSf + (2 + 3 * s) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_kv_full[s], 3 * C::kTileBytes + 3 * kAtomBytes);
        tma_load_3d(st + 0 * C::kTileBytes, &maps.k, &bar_kv_full[s], 0, hk, k0);
        tma_load_3d(st + 1 * C::kTileBytes, &maps.v, &bar_kv_full[s], 0, hk, k0);
        tma_load_3d(st + 2 * C::kTileBytes, &maps.kt, &bar_kv_full[s], 0, hk, k0);
        bulk_load(sf + 0 * kAtomBytes, a.k_sf + katom, kAtomBytes, &bar_kv_full[s]);
        bulk_load(sf + 1 * kAtomBytes, a.v_sf + katom, kAtomBytes, &bar_kv_full[s]);
        bulk_load(sf + 2 * kAtomBytes, a.kt_sf + katom, kAtomBytes, &bar_kv_full[s]);
        issued = j + 1;
      }
      role_wait(&bar_q, 0, abort_flag, nullptr, 0);
      for (int j = (issued > C::kStages ? issued - C::kStages : 0); j < issued; ++j)
        mbar_wait(&bar_kv_full[j % C::kStages], (j / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t qa = smem_u32(smem + C::kOffQ), ga = smem_u32(smem + C::kOffG);
      bool ok = role_wait(&bar_q, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfQ, sSf + 0 * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfG, sSf + 1 * kAtomBytes);
      }
      auto issue_sdp = [&](int j) -> bool {  // S = Q K^T and dP = G V^T, back to back
        const int s = j % C::kStages;
        if (!role_wait(&bar_kv_full[s], (j / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        // S and dP of the previous key tile must have been read out of TMEM
        if (j >= 1 && !role_wait(&bar_x_free, (j - 1) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
        tmem_cp_atom(tmem + C::kSfK + 4 * s, sSf + (2 + 3 * s + 0) * kAtomBytes);
        tmem_cp_atom(tmem + C::kSfV + 4 * s, sSf + (2 + 3 * s + 1) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColS, make_sdesc(qa + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + 32 * kk, 16, C::kSBO, C::kSwz), make_idesc_mxf8(128, 128, 0, 0, kk, kk),
                      tmem + C::kSfQ, tmem + C::kSfK + 4 * s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tmem + C::kColDP, make_sdesc(ga + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_sdesc(st + C::kTileBytes + 32 * kk, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tmem + C::kSfG, tmem + C::kSfV + 4 * s, kk > 0);
        mma_commit(&bar_sdp_full);
        return true;
      };
      if (ok) ok = issue_sdp(0);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int s = j % C::kStages;
        const uint32_t st = smem_u32(smem + C::kOffStage + s * C::kStageBytes);
        if (j + 1 < n_kt && !(ok = issue_sdp(j + 1))) break;  // overlaps the dS work of tile j
        if (!(ok = role_wait(&bar_ds_ready, j & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        tmem_cp_atom(tmem + C::kSfKt + 4 * s, sSf + (2 + 3 * s + 2) * kAtomBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dQ += dS K (contraction over 128 keys)
          mma_mxf8_ts(tmem + C::kColDQ, tmem + C::kColDS + 8 * kk,
                      make_sdesc(st + 2 * C::kTileBytes + kk * 32 * D, 16, C::kSBO, C::kSwz),
                      make_idesc_mxf8(128, D, 0, 1, kk & 1, kk), tmem + (kk < 2 ? C::kSfDS0 : C::kSfDS1),
                      tmem + C::kSfKt + 4 * s, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_ds_free);
        mma_commit(&bar_kv_empty[s]);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    const int quad = warp & 3;
    const int hf = (warp - 4) >> 2;       // column half: keys [64 hf, 64 hf + 64)
    const int r = quad * 32 + lane;       // query row (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t qpos = static_cast<int64_t>(qt) * 128 + r;
    const bool q_valid = qpos < n;
    const int64_t slot = (static_cast<int64_t>(h) * a.ntiles + tile_base + qt) * 128 + r;
    const float nl = -a.lpad[slot];  // -inf for rows past the document end -> P = 0
    const float dd = a.dpad[slot];
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      if (!(ok = warp_wait(&bar_sdp_full, j & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      float p[64];
      tmem_ld64(lane_base + C::kColS + 64 * hf, p);
#pragma unroll
      for (int c = 0; c < 64; ++c) p[c] = ex2_approx(fmaf(p[c], sl2, nl));
      // keys past the document end (last tile) or after the query (diagonal tile)
      const int64_t rem = n - static_cast<int64_t>(j) * 128;
      int lim = rem < 128 ? static_cast<int>(rem) : 128;
      if (a.causal && j == qt) lim = min(lim, r + 1);
      if (lim < 128) {
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = (64 * hf + c < lim) ? p[c] : 0.0f;
      }
      // dS = P (dP - D), in place
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColDP + 64 * hf + 32 * cc, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) p[32 * cc + i] *= (__uint_as_float(rr[i]) - dd);
      }
      tc_fence_before();
      mbar_arrive(&bar_x_free);  // S and dP read: the next tile's S, dP may start
      // the previous dQ MMA must be done with the dS codes and scales
      if (j > 0 && !(ok = warp_wait(&bar_ds_free, (j - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      uint32_t ebytes = 0;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = p[32 * cc + i];
        uint32_t w[8];
        ebytes |= quant_ds_block32(x, 0, w) << (8 * cc);  // 32 query rows x 32 keys
        tmem_st8(lane_base + C::kColDS + 16 * hf + 8 * cc, w);
      }
      // dQ's A operand is dS (rows = queries, groups = 32-key blocks): row r's
      // scales sit in lane r, column base + r / 32; half hf owns key blocks
      // 2 hf, 2 hf + 1.
      tmem_st1(lane_base + (hf ? C::kSfDS1 : C::kSfDS0) + quad, ebytes | 0x7F7F0000u);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
    }
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = doc_start + qpos;
      __nv_bfloat16* dqrow = reinterpret_cast<__nv_bfloat16*>(a.dq_out) + (t * a.Hq + h) * D;
      // each half writes half of the row's channels
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t rr[32];
        const int cb = (D / 2) * hf + 32 * c;
        tmem_ld32(lane_base + C::kColDQ + cb, rr);
        tmem_ld_wait();
        if (q_valid) store_row_bf16(dqrow + cb, rr, a.alpha);
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

cudaError_t launch_bwd_split(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  const int tiles = (max_seqlen + 127) / 128;
  dim3 g1(tiles, a.num_docs, a.Hkv), g2(tiles, a.num_docs, a.Hq);
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkdvCfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqCfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_dkdv_kernel<128><<<g1, kSplitThreads, DkdvCfg<128>::kSmemBytes, stream>>>(m, a);
    attn_bwd_dq_kernel<128><<<g2, kSplitThreads, DqCfg<128>::kSmemBytes, stream>>>(m, a);
  } else {
    e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkdvCfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqCfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_dkdv_kernel<64><<<g1, kSplitThreads, DkdvCfg<64>::kSmemBytes, stream>>>(m, a);
    attn_bwd_dq_kernel<64><<<g2, kSplitThreads, DqCfg<64>::kSmemBytes, stream>>>(m, a);
  }
  return cudaGetLastError();
}

}  // namespace mxa
