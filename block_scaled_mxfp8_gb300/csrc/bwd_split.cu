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
// Warps: 0 = TMA producer, 1 = TMEM owner and MMA issuer, 2..17 = softmax;
// the dK/dV kernel adds warp 18, which issues its gradient MMAs (dV, dK) so
// that the S^T / dP^T issuer never waits behind them.
// Four softmax warps share each TMEM lane quadrant and split the tile's 128
// columns into quarters of 32, so each warp owns exactly one 32 x 32 dS block
// per tile (its block max is a warp reduction) and every SM sub-partition has
// four softmax warps to interleave.  Quarter p writes its block exponent into
// its own scale-factor column block, which the gradient MMA reads for K step
// p.
// LSE (times log2 e; +inf past a document's end) and D come tile-padded from
// the prep kernel and are bulk-loaded with the tiles.
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace mxa {

namespace {

constexpr int kSplitThreads = 576;
constexpr int kDkdvThreads = 608;  // + warp 18, the gradient-MMA issuer
constexpr int kSoftmaxThreads = 512;

template <int D>
struct DkdvCfg {
  // ring A (Q, G tiles, LSE row) feeds S^T and dP^T and is released after
  // dP^T; ring B (Qt, Gt tiles, D row) feeds dV and dK and is released after
  // dK, so the next units' Q and G load while the gradient MMAs still run
  static constexpr int kStagesA = 3, kStagesB = 2;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  // TMEM: X holds S^T then dP^T; dV, dK accumulators; P^T and dS^T codes;
  // scale slots indexed by unit parity (+4 (u & 1))
  static constexpr uint32_t kColX = 0, kColDV = 128, kColDK = 256, kColP = 384, kColDS = 416;
  static constexpr uint32_t kSfK = 448, kSfQ = 452 /*+4t*/, kSfV = 460, kSfG = 464 /*+4t*/, kSfP = 472,
                            kSfGt = 476 /*+4t*/, kSfQt = 484 /*+4t*/, kSfDS = 492 /*+4 per query block*/;
  // shared memory: K, V, ring A stages (Q, G), ring B stages (Qt, Gt), the
  // LSE and D rows of the stages, then the scale atoms
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffA = kOffV + kTileBytes;
  static constexpr int kOffB = kOffA + kStagesA * 2 * kTileBytes;
  static constexpr int kOffRowsA = kOffB + kStagesB * 2 * kTileBytes;  // LSE rows, 512 B each
  static constexpr int kOffRowsB = kOffRowsA + kStagesA * 512;         // D rows
  static constexpr int kOffSf = kOffRowsB + kStagesB * 512;  // K, V, then 2 per A stage, 2 per B stage
  // staging of the dS codes emitted for the dQ product: the 128 x 128 tile as
  // the 128-byte-swizzled image a TMA load would produce, stored with one bulk
  // copy and read back by the dQ kernel with one bulk copy
  static constexpr int kOffDsStage = (kOffSf + (2 + 2 * kStagesA + 2 * kStagesB) * kAtomBytes + 1023) & ~1023;
  static constexpr int kSmemBytes = kOffDsStage + 16384 + 1024;
};

template <int D>
struct DqCfg {
  // ring A (K, V tiles) feeds S and dP and is released once they complete;
  // ring B (Kt tiles) feeds dQ
  static constexpr int kStagesA = 3, kStagesB = 3;
  static constexpr int kTileBytes = 128 * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;
  // TMEM: S and dP side by side (both MMAs issue back to back), dQ
  // accumulator, dS codes and scales double-buffered by tile parity (t = j & 1)
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384 /*+32t*/;
  static constexpr uint32_t kSfQ = 448, kSfG = 452, kSfK = 456 /*+4t*/, kSfV = 464 /*+4t*/,
                            kSfDS = 472 /*+16t, +4 per key block*/, kSfKt = 504 /*+4t*/;
  static constexpr int kOffQ = 0;
  static constexpr int kOffG = kOffQ + kTileBytes;
  static constexpr int kOffA = kOffG + kTileBytes;                     // per A stage: K, V
  static constexpr int kOffB = kOffA + kStagesA * 2 * kTileBytes;      // per B stage: Kt
  static constexpr int kOffSf = kOffB + kStagesB * kTileBytes;         // Q, G, 2 per A stage, 1 per B stage
  static constexpr int kSmemBytes = kOffSf + (2 + 2 * kStagesA + kStagesB) * kAtomBytes + 1024;
};

template <int kCount = 32>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&rr)[32], float mul) {
#pragma unroll
  for (int i = 0; i < kCount; i += 8) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(rr[i]) * mul, __uint_as_float(rr[i + 1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * mul, __uint_as_float(rr[i + 3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * mul, __uint_as_float(rr[i + 5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * mul, __uint_as_float(rr[i + 7]) * mul);
    *reinterpret_cast<uint4*>(dst + i) = v;
  }
}

}  // namespace

// ========================================================================= dK, dV
// ORDER (causal calls over equal documents, without a tile list): the launch
// order of causal_launch_order, heaviest key tiles of the last groups first
// (the other calls keep the grid's own order and this code out of their build).
template <int D, bool STRICT, bool ORDER>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_kv, bar_a_full[C::kStagesA], bar_a_empty[C::kStagesA], bar_b_full[C::kStagesB],
      bar_b_empty[C::kStagesB], bar_s_full, bar_x_free, bar_dp_full, bar_x_free2, bar_p_ready, bar_ds_ready,
      bar_dv_done, bar_dk_done, bar_final, bar_drain, bar_drain2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot, s_slot_k;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int kt, b, hk;
  int64_t ktile_base = -1, tile_base = -1;  // first scale tiles of the document: keys, queries
  if (a.k_items) {
    if (!list_item(a.k_items, a.k_count, a.Hkv, b, hk, kt, ktile_base, tile_base)) return;
  } else {
    kt = blockIdx.x;
    b = blockIdx.y;
    hk = blockIdx.z;
    if constexpr (ORDER) {
      // key tile kt carries (tiles - kt) units
      const int v = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
      int g;
      causal_launch_order(v, a.num_docs * a.Hkv, static_cast<int>(gridDim.x), g, kt);
      b = g % a.num_docs;
      hk = g / a.num_docs;
    }
  }
  const int grp = a.Hq / a.Hkv;
  int64_t doc_start, n, kdoc_start, nk;  // the document's queries and keys (the same for self-attention)
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  doc_bounds(a.cu_k, a.num_docs, a.Tk, b, kdoc_start, nk);
  const int n_tiles = static_cast<int>((n + 127) / 128);  // query tiles
  if (static_cast<int64_t>(kt) * 128 >= nk) return;
  const int qi0 = a.causal ? kt : 0;
  const int nq = n_tiles > qi0 ? n_tiles - qi0 : 0;
  const int n_work = nq * grp;
  if (tile_base < 0) tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, kDkdvThreads, &s_slot);
  if (ktile_base < 0)
    ktile_base = (a.cu_k == a.cu_seqlens && a.Tk == a.T) ? tile_base
                                                          : doc_tile_base(a.cu_k, b, nk, tid, kDkdvThreads, &s_slot_k);

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(&bar_a_full[s], 1);
      mbar_init(&bar_a_empty[s], 1 + kSoftmaxThreads / 32);  // dP^T commit + one lane per softmax warp
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(&bar_b_full[s], 1);
      mbar_init(&bar_b_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_x_free, kSoftmaxThreads);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_x_free2, kSoftmaxThreads);
    mbar_init(&bar_p_ready, kSoftmaxThreads);
    mbar_init(&bar_ds_ready, kSoftmaxThreads);
    mbar_init(&bar_dv_done, 1);
    mbar_init(&bar_dk_done, 1);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_drain2, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  uint8_t* sSf = smem + C::kOffSf;  // [0] K, [1] V, A stage s: 2 + 2s (Q, G), B stage s: 2 + 2 kStagesA + 2s (Qt, Gt)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const int64_t k0 = kdoc_start + static_cast<int64_t>(kt) * 128;
      const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + kt) * kAtomBytes;
      mbar_arrive_expect_tx(&bar_kv, 2 * C::kTileBytes + 2 * kAtomBytes);
      tma_load_3d(smem + C::kOffK, &maps.k, &bar_kv, 0, hk, static_cast<int>(k0));
      tma_load_3d(smem + C::kOffV, &maps.v, &bar_kv, 0, hk, static_cast<int>(k0));
      bulk_load(sSf + 0 * kAtomBytes, a.k_sf + katom, kAtomBytes, &bar_kv);
      bulk_load(sSf + 1 * kAtomBytes, a.v_sf + katom, kAtomBytes, &bar_kv);
      int issued_a = 0, issued_b = 0;
      for (int u = 0; u < n_work; ++u) {
        const int sa = u % C::kStagesA, sb = u % C::kStagesB;
        const int h = hk * grp + u / nq;
        const int qi = qi0 + u % nq;
        const int q0 = static_cast<int>(doc_start + static_cast<int64_t>(qi) * 128);
        const int64_t qslot = static_cast<int64_t>(h) * a.ntiles + tile_base + qi;
        if (u >= C::kStagesA &&
            !role_wait(&bar_a_empty[sa], ((u / C::kStagesA) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        uint8_t* st = smem + C::kOffA + sa * 2 * C::kTileBytes;
        uint8_t* sf = sSf + (2 + 2 * sa) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_a_full[sa], 2 * C::kTileBytes + 2 * kAtomBytes + 512);
        tma_load_3d(st, &maps.q, &bar_a_full[sa], 0, h, q0);
        tma_load_3d(st + C::kTileBytes, &maps.g, &bar_a_full[sa], 0, h, q0);
        bulk_load(smem + C::kOffRowsA + sa * 512, a.lpad + qslot * 128, 512, &bar_a_full[sa]);
        bulk_load(sf, a.q_sf + qslot * kAtomBytes, kAtomBytes, &bar_a_full[sa]);
        bulk_load(sf + kAtomBytes, a.g_sf + qslot * kAtomBytes, kAtomBytes, &bar_a_full[sa]);
        issued_a = u + 1;
        if (u >= C::kStagesB &&
            !role_wait(&bar_b_empty[sb], ((u / C::kStagesB) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        st = smem + C::kOffB + sb * 2 * C::kTileBytes;
        sf = sSf + (2 + 2 * C::kStagesA + 2 * sb) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_b_full[sb], 2 * C::kTileBytes + 2 * kAtomBytes + 512);
        tma_load_3d(st, &maps.qt, &bar_b_full[sb], 0, h, q0);
        tma_load_3d(st + C::kTileBytes, &maps.gt, &bar_b_full[sb], 0, h, q0);
        bulk_load(smem + C::kOffRowsB + sb * 512, a.dpad + qslot * 128, 512, &bar_b_full[sb]);
        bulk_load(sf, a.qt_sf + qslot * kAtomBytes, kAtomBytes, &bar_b_full[sb]);
        bulk_load(sf + kAtomBytes, a.gt_sf + qslot * kAtomBytes, kAtomBytes, &bar_b_full[sb]);
        issued_b = u + 1;
      }
      role_wait(&bar_kv, 0, abort_flag, nullptr, 0);
      for (int u = (issued_a > C::kStagesA ? issued_a - C::kStagesA : 0); u < issued_a; ++u)
        mbar_wait(&bar_a_full[u % C::kStagesA], (u / C::kStagesA) & 1, nullptr, 0);
      for (int u = (issued_b > C::kStagesB ? issued_b - C::kStagesB : 0); u < issued_b; ++u)
        mbar_wait(&bar_b_full[u % C::kStagesB], (u / C::kStagesB) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- S^T / dP^T issuer
      // descriptors built once; per MMA only constant offsets are added
      const uint64_t dKa = make_sdesc(smem_u32(smem + C::kOffK), 16, C::kSBO, C::kSwz);
      const uint64_t dVa = make_sdesc(smem_u32(smem + C::kOffV), 16, C::kSBO, C::kSwz);
      const uint64_t dA = make_sdesc(smem_u32(smem + C::kOffA), 16, C::kSBO, C::kSwz);
      const uint64_t dSf = atom_desc(sSf);
      const uint32_t tX = tmem + C::kColX;
      const uint32_t tSfK = tmem + C::kSfK, tSfV = tmem + C::kSfV;
      bool ok = role_wait(&bar_kv, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_desc(tSfK, dSf);
        tmem_cp_desc(tSfV, sdesc_adv(dSf, kAtomBytes));
      }
      auto issue_s = [&](int u) -> bool {  // S^T = K Q^T into X
        const int sa = u % C::kStagesA;
        if (!role_wait(&bar_a_full[sa], (u / C::kStagesA) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint64_t dq = sdesc_adv(dA, sa * 2 * C::kTileBytes);
        const uint32_t tSfQ = tmem + C::kSfQ + 4 * (u & 1);
        tmem_cp_desc(tSfQ, sdesc_adv(dSf, (2 + 2 * sa) * kAtomBytes));
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tX, sdesc_adv(dKa, 32 * kk), sdesc_adv(dq, 32 * kk), make_idesc_mxf8(128, 128, 0, 0, kk, kk),
                      tSfK, tSfQ, kk > 0);
        mma_commit(&bar_s_full);
        return true;
      };
      // Per unit u: dP^T_u once S^T_u has been read out of X, then S^T_{u+1}
      // once dP^T_u has been read; warp 18 issues the gradient MMAs.
      if (ok && n_work > 0) ok = issue_s(0);
      for (int u = 0; ok && u < n_work; ++u) {
        const int sa = u % C::kStagesA, sb = u % C::kStagesB, t = u & 1;
        const uint64_t da = sdesc_adv(dA, sa * 2 * C::kTileBytes);  // Q, G of this unit
        // dP^T = V G^T; ring B (its D row) must have landed before the
        // softmax warps see dP^T
        if (!(ok = role_wait(&bar_x_free, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (!(ok = role_wait(&bar_b_full[sb], (u / C::kStagesB) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        const uint32_t tSfG = tmem + C::kSfG + 4 * t;
        tmem_cp_desc(tSfG, sdesc_adv(dSf, (2 + 2 * sa + 1) * kAtomBytes));
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tX, sdesc_adv(dVa, 32 * kk), sdesc_adv(da, C::kTileBytes + 32 * kk),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tSfV, tSfG, kk > 0);
        mma_commit(&bar_dp_full);
        mma_commit(&bar_a_empty[sa]);
        // next S^T as soon as dP^T has been read (runs while dS is formed)
        if (!(ok = role_wait(&bar_x_free2, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (u + 1 < n_work && !(ok = issue_s(u + 1))) break;
      }
      // drain this thread's MMAs before the TMEM is released
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp == 18) {
    if (lane == 0) {
      // ---------------------------------------------------------- dV / dK issuer
      const uint64_t dB = make_sdesc(smem_u32(smem + C::kOffB), 16, C::kSBO, C::kSwz);
      const uint64_t dSf = atom_desc(sSf);
      const uint32_t tDV = tmem + C::kColDV, tDK = tmem + C::kColDK;
      const uint32_t tP = tmem + C::kColP, tDS = tmem + C::kColDS;
      const uint32_t tSfP = tmem + C::kSfP, tSfDS = tmem + C::kSfDS;
      bool ok = true;
      for (int u = 0; u < n_work; ++u) {
        const int sb = u % C::kStagesB, t = u & 1;
        const uint64_t db = sdesc_adv(dB, sb * 2 * C::kTileBytes);  // Qt, Gt of this unit
        // dV += P^T G once the softmax warps have written P^T and ring B has
        // landed
        if (!(ok = role_wait(&bar_p_ready, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (!(ok = role_wait(&bar_b_full[sb], (u / C::kStagesB) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        const uint32_t tSfGt = tmem + C::kSfGt + 4 * t;
        tmem_cp_desc(tSfGt, sdesc_adv(dSf, (2 + 2 * C::kStagesA + 2 * sb + 1) * kAtomBytes));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf8_ts(tDV, tP + 8 * kk, sdesc_adv(db, C::kTileBytes + kk * 32 * D),
                      make_idesc_mxf8(128, D, 0, 1, kk, kk), tSfP, tSfGt, (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_dv_done);
        // dK += dS^T Q once dS^T is in TMEM (and its copy staged)
        if (!(ok = role_wait(&bar_ds_ready, u & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (a.ds_codes) {  // the staged dS tile of this unit to the workspace
          const int h = hk * grp + u / nq;
          const int64_t pair = (static_cast<int64_t>(h) * a.ntiles_k + ktile_base + kt) * a.mt + (qi0 + u % nq);
          bulk_store(a.ds_codes + pair * 16384, smem + C::kOffDsStage, 16384);
        }
        tc_fence_after();
        const uint32_t tSfQt = tmem + C::kSfQt + 4 * t;
        tmem_cp_desc(tSfQt, sdesc_adv(dSf, (2 + 2 * C::kStagesA + 2 * sb) * kAtomBytes));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_mxf8_ts(tDK, tDS + 8 * kk, sdesc_adv(db, kk * 32 * D), make_idesc_mxf8(128, D, 0, 1, 0, kk),
                      tSfDS + 4 * kk, tSfQt, (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_b_empty[sb]);
        // the staging buffer is free for the next unit's dS once the bulk
        // store has read it; dk_done tells the softmax warps both
        if (a.ds_codes) bulk_store_wait_read();
        mma_commit(&bar_dk_done);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain2);
      mbar_wait(&bar_drain2, 0, nullptr, 0);
      if (a.ds_codes) bulk_store_wait_all();  // the last staged tile is out before the CTA exits
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / dS
    // Warp w serves TMEM lane quadrant w % 4 (key rows) and query columns
    // [32 part, 32 part + 32): one 32 x 32 block of P^T and dS^T per unit.
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
    const int j = quad * 32 + lane;       // key row (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t kpos = static_cast<int64_t>(kt) * 128 + j;
    const bool key_valid = kpos < nk;
    const float kb8 = key_valid ? 8.0f : -INFINITY;  // 2^8 boost of P^T; invalid key rows -> 0
    const float sl2 = a.scale_log2;
    const uint64_t kb8x2 = f2_pack(kb8, kb8), sl2x2 = f2_pack(sl2, sl2);
    if (part == 0) {
      tmem_st4(lane_base + C::kSfP, 0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);  // 2^-8
      tmem_st_wait();
    }
    bool ok = true;
    // strict dQ: 2^e_k of this thread's key (the K fold of the diagonal pair)
    float kfold = 1.0f;
    if constexpr (STRICT) {
      if (key_valid) {
        const uint32_t kb = a.kkey_sf[(static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + kt) * 128 + j];
        kfold = kb ? __uint_as_float(kb << 23) : __uint_as_float(0x00400000u);
      }
    }
    for (int u = 0; u < n_work; ++u) {
      const int sa = u % C::kStagesA, sb = u % C::kStagesB;
      const int qi = qi0 + u % nq;
      const float* lrow = reinterpret_cast<const float*>(smem + C::kOffRowsA + sa * 512) + 32 * part;
      const float* drow = reinterpret_cast<const float*>(smem + C::kOffRowsB + sb * 512) + 32 * part;
      if (!(ok = warp_wait(&bar_s_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      float p[32];
      {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColX + 32 * part, rr);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) p[c] = __uint_as_float(rr[c]);
      }
      tc_fence_before();
      mbar_arrive(&bar_x_free);
      // P^T boosted by 2^8 (P <= 1 after the LSE normalization); rows past the
      // document end have LSE = +inf, so their P is 0 without a test
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lrow + c);
        const float2 a = f2_unpack(f2_fma(f2_pack(p[c], p[c + 1]), sl2x2, f2_sub(kb8x2, f2_pack(l4.x, l4.y))));
        const float2 b = f2_unpack(f2_fma(f2_pack(p[c + 2], p[c + 3]), sl2x2, f2_sub(kb8x2, f2_pack(l4.z, l4.w))));
        p[c] = ex2_approx(a.x);
        p[c + 1] = ex2_approx(a.y);
        p[c + 2] = ex2_approx(b.x);
        p[c + 3] = ex2_approx(b.y);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_a_empty[sa]);  // this warp is done with the LSE row
      if (a.causal && qi == kt) {  // diagonal tile: query index (in tile) >= key index
#pragma unroll
        for (int c = 0; c < 32; ++c) p[c] = (32 * part + c >= j) ? p[c] : 0.0f;
      }
      // the previous unit's dV MMA must be done with the P^T codes
      if (u > 0 && !(ok = warp_wait(&bar_dv_done, (u - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = pack_e4m3x4(p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]);
        tmem_st8(lane_base + C::kColP + 8 * part, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p_ready);
      if (!(ok = warp_wait(&bar_dp_full, u & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      // dS^T = P^T (dP^T - D), in place
      {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColX + 32 * part, rr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bar_x_free2);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(drow + i);
          const float2 a = f2_unpack(f2_mul(f2_pack(p[i], p[i + 1]),
                                            f2_sub(f2_pack(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])),
                                                   f2_pack(d4.x, d4.y))));
          const float2 b = f2_unpack(f2_mul(f2_pack(p[i + 2], p[i + 3]),
                                            f2_sub(f2_pack(__uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3])),
                                                   f2_pack(d4.z, d4.w))));
          p[i] = a.x;
          p[i + 1] = a.y;
          p[i + 2] = b.x;
          p[i + 3] = b.y;
        }
      }
      {
        uint32_t w[8];
        const uint32_t eb = quant_ds_block32(p, 8, w);  // 32 key rows x 32 queries
        // the previous unit's dK MMA must be done with the dS^T codes and
        // scales, and its bulk store with the staging buffer
        if (u > 0 && !(ok = warp_wait(&bar_dk_done, (u - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        tmem_st8(lane_base + C::kColDS + 8 * part, w);
        // dK's A operand is dS^T (rows = keys, K = queries): for K step
        // `part` the scale of row r sits in lane r, column kSfDS + 4 part +
        // r / 32, byte 0
        tmem_st1(lane_base + C::kSfDS + 4 * part + quad, eb | 0x7F7F7F00u);
        if (a.ds_codes) {
          // the same block for the dQ product: codes of key row j, queries
          // [32 part, 32 part + 32) -- 16-byte chunks 2 part, 2 part + 1 of
          // the row, placed at chunk ^ (j & 7) (the 128-byte swizzle); its
          // scale byte at 4 part + quad of the pair's 16 (query block major)
          const int h = hk * grp + u / nq;
          const int64_t pair = (static_cast<int64_t>(h) * a.ntiles_k + ktile_base + kt) * a.mt + qi;
          uint32_t we[8];
          if constexpr (STRICT) {
            // strict dQ: one scale per query (column c) over the block's 32
            // keys, after the diagonal pair's K fold; lane c keeps query c's
            const uint8_t eq = quant_ds_cols32(p, 8, (a.causal && qi == kt) ? kfold : 1.0f, lane, we);
            a.ds_sf[pair * 512 + lane * 16 + part * 4 + quad] = eq;
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) we[k] = w[k];
            if (lane == 0) a.ds_sf[pair * 16 + part * 4 + quad] = static_cast<uint8_t>(eb);
          }
          uint8_t* row = smem + C::kOffDsStage + j * 128;
          *reinterpret_cast<uint4*>(row + (((2 * part) ^ (j & 7)) << 4)) = make_uint4(we[0], we[1], we[2], we[3]);
          *reinterpret_cast<uint4*>(row + (((2 * part + 1) ^ (j & 7)) << 4)) = make_uint4(we[4], we[5], we[6], we[7]);
          fence_proxy_async_smem();  // the MMA thread's bulk store reads it
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
    }
    // ---------------------------------------------------------- dK, dV out
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = kdoc_start + kpos;
      __nv_bfloat16* dvrow = reinterpret_cast<__nv_bfloat16*>(a.dv) + (t * a.Hkv + hk) * D;
      __nv_bfloat16* dkrow = reinterpret_cast<__nv_bfloat16*>(a.dk) + (t * a.Hkv + hk) * D;
      // each warp writes D/4 channels of dV and of dK for its key rows
      constexpr int kCols = D / 4;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t col = (g ? C::kColDK : C::kColDV) + kCols * part;
        __nv_bfloat16* dst = (g ? dkrow : dvrow) + kCols * part;
        const float mul = g ? a.alpha : 1.0f;
        uint32_t rr[32];
        if constexpr (kCols == 32) {
          tmem_ld32(lane_base + col, rr);
        } else {
          uint32_t r16[16];
          tmem_ld16(lane_base + col, r16);
#pragma unroll
          for (int i = 0; i < 16; ++i) rr[i] = r16[i];
        }
        tmem_ld_wait();
        if (n_work == 0) {  // a document with keys but no queries: zero gradients
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (key_valid) store_row_bf16<kCols>(dst, rr, mul);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

  __shared__ uint64_t bar_q, bar_a_full[C::kStagesA], bar_a_empty[C::kStagesA], bar_b_full[C::kStagesB],
      bar_b_empty[C::kStagesB], bar_sdp_full, bar_x_free, bar_ds_ready, bar_final, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot, s_slot_k;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int b, h, qt;
  int64_t tile_base = -1, ktile_base = -1;  // first scale tiles of the document: queries, keys
  if (a.q_items) {
    if (!list_item(a.q_items, a.q_count, a.Hq, b, h, qt, tile_base, ktile_base)) return;
  } else {
    b = blockIdx.y;
    h = blockIdx.z;
    qt = a.causal ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  }
  const int hk = h / (a.Hq / a.Hkv);
  int64_t doc_start, n, kdoc_start, nk;  // the document's queries and keys
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  doc_bounds(a.cu_k, a.num_docs, a.Tk, b, kdoc_start, nk);
  const int n_tiles = static_cast<int>((n + 127) / 128);
  if (qt >= n_tiles) return;
  const int n_kt = a.causal ? qt + 1 : static_cast<int>((nk + 127) / 128);
  if (tile_base < 0) tile_base = doc_tile_base(a.cu_seqlens, b, n, tid, kSplitThreads, &s_slot);
  if (ktile_base < 0)
    ktile_base = (a.cu_k == a.cu_seqlens && a.Tk == a.T) ? tile_base
                                                          : doc_tile_base(a.cu_k, b, nk, tid, kSplitThreads, &s_slot_k);

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < C::kStagesA; ++s) {
      mbar_init(&bar_a_full[s], 1);
      mbar_init(&bar_a_empty[s], 1);
    }
    for (int s = 0; s < C::kStagesB; ++s) {
      mbar_init(&bar_b_full[s], 1);
      mbar_init(&bar_b_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_x_free, kSoftmaxThreads);
    mbar_init(&bar_ds_ready, kSoftmaxThreads);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  uint8_t* sSf = smem + C::kOffSf;  // [0] Q, [1] G, A stage s: 2 + 2s (K, V), B stage s: 2 + 2 kStagesA + s (Kt)

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
      int issued_a = 0, issued_b = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int sa = j % C::kStagesA, sb = j % C::kStagesB;
        const int k0 = static_cast<int>(kdoc_start + static_cast<int64_t>(j) * 128);
        const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + j) * kAtomBytes;
        if (j >= C::kStagesA &&
            !role_wait(&bar_a_empty[sa], ((j / C::kStagesA) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        uint8_t* st = smem + C::kOffA + sa * 2 * C::kTileBytes;
        uint8_t* sf = sSf + (2 + 2 * sa) * kAtomBytes;
        mbar_arrive_expect_tx(&bar_a_full[sa], 2 * C::kTileBytes + 2 * kAtomBytes);
        tma_load_3d(st, &maps.k, &bar_a_full[sa], 0, hk, k0);
        tma_load_3d(st + C::kTileBytes, &maps.v, &bar_a_full[sa], 0, hk, k0);
        bulk_load(sf, a.k_sf + katom, kAtomBytes, &bar_a_full[sa]);
        bulk_load(sf + kAtomBytes, a.v_sf + katom, kAtomBytes, &bar_a_full[sa]);
        issued_a = j + 1;
        if (j >= C::kStagesB &&
            !role_wait(&bar_b_empty[sb], ((j / C::kStagesB) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        mbar_arrive_expect_tx(&bar_b_full[sb], C::kTileBytes + kAtomBytes);
        tma_load_3d(smem + C::kOffB + sb * C::kTileBytes, &maps.kt, &bar_b_full[sb], 0, hk, k0);
        bulk_load(sSf + (2 + 2 * C::kStagesA + sb) * kAtomBytes, a.kt_sf + katom, kAtomBytes, &bar_b_full[sb]);
        issued_b = j + 1;
      }
      role_wait(&bar_q, 0, abort_flag, nullptr, 0);
      for (int j = (issued_a > C::kStagesA ? issued_a - C::kStagesA : 0); j < issued_a; ++j)
        mbar_wait(&bar_a_full[j % C::kStagesA], (j / C::kStagesA) & 1, nullptr, 0);
      for (int j = (issued_b > C::kStagesB ? issued_b - C::kStagesB : 0); j < issued_b; ++j)
        mbar_wait(&bar_b_full[j % C::kStagesB], (j / C::kStagesB) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint64_t dQa = make_sdesc(smem_u32(smem + C::kOffQ), 16, C::kSBO, C::kSwz);
      const uint64_t dGa = make_sdesc(smem_u32(smem + C::kOffG), 16, C::kSBO, C::kSwz);
      const uint64_t dA = make_sdesc(smem_u32(smem + C::kOffA), 16, C::kSBO, C::kSwz);
      const uint64_t dB = make_sdesc(smem_u32(smem + C::kOffB), 16, C::kSBO, C::kSwz);
      const uint64_t dSf = atom_desc(sSf);
      const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tDQ = tmem + C::kColDQ, tDS = tmem + C::kColDS;
      const uint32_t tSfQ = tmem + C::kSfQ, tSfG = tmem + C::kSfG;
      const uint32_t tSfDS = tmem + C::kSfDS;
      bool ok = role_wait(&bar_q, 0, abort_flag, a.err, kErrTimeoutMma);
      if (ok) {
        tc_fence_after();
        tmem_cp_desc(tSfQ, dSf);
        tmem_cp_desc(tSfG, sdesc_adv(dSf, kAtomBytes));
      }
      auto issue_sdp = [&](int j) -> bool {  // S = Q K^T and dP = G V^T, back to back
        const int sa = j % C::kStagesA;
        if (!role_wait(&bar_a_full[sa], (j / C::kStagesA) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        // S and dP of the previous key tile must have been read out of TMEM
        if (j >= 1 && !role_wait(&bar_x_free, (j - 1) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint64_t dstage = sdesc_adv(dA, sa * 2 * C::kTileBytes);  // K, V
        const uint64_t dsf = sdesc_adv(dSf, (2 + 2 * sa) * kAtomBytes);
        const uint32_t tSfK = tmem + C::kSfK + 4 * (j & 1), tSfV = tmem + C::kSfV + 4 * (j & 1);
        tmem_cp_desc(tSfK, dsf);
        tmem_cp_desc(tSfV, sdesc_adv(dsf, kAtomBytes));
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tS, sdesc_adv(dQa, 32 * kk), sdesc_adv(dstage, 32 * kk), make_idesc_mxf8(128, 128, 0, 0, kk, kk),
                      tSfQ, tSfK, kk > 0);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tDP, sdesc_adv(dGa, 32 * kk), sdesc_adv(dstage, C::kTileBytes + 32 * kk),
                      make_idesc_mxf8(128, 128, 0, 0, kk, kk), tSfG, tSfV, kk > 0);
        mma_commit(&bar_sdp_full);
        mma_commit(&bar_a_empty[sa]);
        return true;
      };
      if (ok && n_kt > 0) ok = issue_sdp(0);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int sb = j % C::kStagesB;
        if (j + 1 < n_kt && !(ok = issue_sdp(j + 1))) break;  // overlaps the dS work of tile j
        if (!(ok = role_wait(&bar_ds_ready, j & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (!(ok = role_wait(&bar_b_full[sb], (j / C::kStagesB) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        const uint32_t tSfKt = tmem + C::kSfKt + 4 * (j & 1);
        tmem_cp_desc(tSfKt, sdesc_adv(dSf, (2 + 2 * C::kStagesA + sb) * kAtomBytes));
        const uint64_t dkt = sdesc_adv(dB, sb * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dQ += dS K (contraction over 128 keys)
          mma_mxf8_ts(tDQ, tDS + 32 * (j & 1) + 8 * kk, sdesc_adv(dkt, kk * 32 * D),
                      make_idesc_mxf8(128, D, 0, 1, 0, kk), tSfDS + 16 * (j & 1) + 4 * kk, tSfKt,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_b_empty[sb]);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax / dS
    // Warp w serves TMEM lane quadrant w % 4 (query rows) and key columns
    // [32 part, 32 part + 32): one 32 x 32 block of P and dS per key tile.
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
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
      float p[32];
      {
        uint32_t rs[32], rd[32];
        tmem_ld32(lane_base + C::kColS + 32 * part, rs);
        tmem_ld32(lane_base + C::kColDP + 32 * part, rd);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bar_x_free);  // S and dP read: the next tile's S, dP may start
        // keys past the document end (last tile) or after the query (diagonal tile)
        const int64_t rem = nk - static_cast<int64_t>(j) * 128;
        int lim = rem < 128 ? static_cast<int>(rem) : 128;
        if (a.causal && j == qt) lim = min(lim, r + 1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float pc = ex2_approx(fmaf(__uint_as_float(rs[c]), sl2, nl));
          // dS = P (dP - D)
          p[c] = (32 * part + c < lim) ? pc * (__uint_as_float(rd[c]) - dd) : 0.0f;
        }
      }
      // dS codes and scales alternate between two TMEM buffers: dQ_{j-2},
      // the last reader of this buffer, was issued before S_j and dP_j, so
      // sdp_full(j) has completed only after it
      {
        const uint32_t t = j & 1;
        uint32_t w[8];
        const uint32_t eb = quant_ds_block32(p, 0, w);  // 32 query rows x 32 keys
        tmem_st8(lane_base + C::kColDS + 32 * t + 8 * part, w);
        // dQ's A operand is dS (rows = queries, K = keys): for K step `part`
        // the scale of row r sits in lane r, column kSfDS + 16 t + 4 part + r / 32
        tmem_st1(lane_base + C::kSfDS + 16 * t + 4 * part + quad, eb | 0x7F7F7F00u);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
    }
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = doc_start + qpos;
      __nv_bfloat16* dqrow = reinterpret_cast<__nv_bfloat16*>(a.dq_out) + (t * a.Hq + h) * D;
      // each warp writes D/4 channels of the row
      constexpr int kCols = D / 4;
      uint32_t rr[32];
      if constexpr (kCols == 32) {
        tmem_ld32(lane_base + C::kColDQ + kCols * part, rr);
      } else {
        uint32_t r16[16];
        tmem_ld16(lane_base + C::kColDQ + kCols * part, r16);
#pragma unroll
        for (int i = 0; i < 16; ++i) rr[i] = r16[i];
      }
      tmem_ld_wait();
      if (q_valid) store_row_bf16<kCols>(dqrow + kCols * part, rr, a.alpha);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

namespace {

template <int D, bool STRICT, bool ORDER>
cudaError_t launch_dkdv_t(const BwdArgs& a, const BwdMaps& m, const dim3& g1, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, STRICT, ORDER>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<D, STRICT, ORDER><<<g1, kDkdvThreads, DkdvCfg<D>::kSmemBytes, stream>>>(m, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& a, const BwdMaps& m, const dim3& g1, cudaStream_t stream) {
  const bool strict = a.kkey_sf != nullptr;
  const bool order = a.causal && !a.k_items && a.cu_seqlens == nullptr && a.cu_k == nullptr;
  if (strict) return order ? launch_dkdv_t<D, true, true>(a, m, g1, stream) : launch_dkdv_t<D, true, false>(a, m, g1, stream);
  return order ? launch_dkdv_t<D, false, true>(a, m, g1, stream) : launch_dkdv_t<D, false, false>(a, m, g1, stream);
}

cudaError_t launch_dkdv(const BwdArgs& a, const BwdMaps& m, int d, const dim3& g1, cudaStream_t stream) {
  return d == 128 ? launch_dkdv_d<128>(a, m, g1, stream) : launch_dkdv_d<64>(a, m, g1, stream);
}

}  // namespace

cudaError_t launch_bwd_split(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  const int tiles = (max_seqlen + 127) / 128;
  const dim3 g1 = a.k_items ? dim3(static_cast<unsigned>(a.ntiles_k * a.Hkv)) : dim3(tiles, a.num_docs, a.Hkv);
  const dim3 g2 = a.q_items ? dim3(static_cast<unsigned>(a.ntiles * a.Hq)) : dim3(tiles, a.num_docs, a.Hq);
  cudaError_t e = launch_dkdv(a, m, d, g1, stream);
  if (e != cudaSuccess) return e;
  if (d == 128) {
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqCfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_dq_kernel<128><<<g2, kSplitThreads, DqCfg<128>::kSmemBytes, stream>>>(m, a);
  } else {
    e = cudaFuncSetAttribute(attn_bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DqCfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_bwd_dq_kernel<64><<<g2, kSplitThreads, DqCfg<64>::kSmemBytes, stream>>>(m, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_emit(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  const int tiles = (max_seqlen + 127) / 128;
  const dim3 g1 = a.k_items ? dim3(static_cast<unsigned>(a.ntiles_k * a.Hkv)) : dim3(tiles, a.num_docs, a.Hkv);
  const cudaError_t e = launch_dkdv(a, m, d, g1, stream);
  if (e != cudaSuccess) return e;
  return launch_dq_gemm(a, m, d, max_seqlen, stream);
}

}  // namespace mxa
