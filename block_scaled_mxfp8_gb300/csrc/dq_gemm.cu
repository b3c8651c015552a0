// dq_gemm.cu -- dQ = alpha * dS K over the dS blocks the dK/dV kernel emitted.
//
// FLAMIA notes, Algorithm 1 step 14 (dQ_i += dS_ij K_j), with dS taken from
// where it was formed once: the dK/dV kernel quantizes every 32 x 32 dS block
// (FA4 write-up, "Квантование dS без транспонирования") and stores its E4M3
// codes plus one UE8M0 scale per block.  The dQ product is then a plain
// block-scaled GEMM per (128-query tile, query head, document), summed over
// the visible key tiles in TMEM in a fixed order (deterministic, no atomics):
//   A = dS   [128 queries x 128 keys]: the stored tile has key rows of query
//            bytes, i.e. an MN-major A operand, kept as the image of its
//            128-byte-swizzled shared-memory layout so that one bulk copy
//            loads it; its 16 block scales come as 16 bytes per tile pair and
//            the epilogue warps (idle until the end) spread them into the
//            scale-factor layout in TMEM, each warp its quarter of the query
//            rows;
//   B = K    TOK view (rows = channels, groups = 32-key blocks), MN-major.
// Warps: 0 = TMA producer, 1 = TMEM owner and MMA issuer, 2..5 = epilogue.
//
// FP16 x 2^9 dQ mode (F16): the FA4 write-up's reduced-precision dQ sum --
// every key tile's partial product is rounded to fp16 after a 2^9 boost (and
// alpha) and added to an fp16 sum, RNE at each step, then brought back by
// 2^-9.  Here the partial of key tile j lands in TMEM (the MMAs of each tile
// start a fresh accumulation), the epilogue warps fold it into their fp16
// registers in key-tile order and hand the columns back before tile j + 1
// overwrites them.
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace mxa {

namespace {

template <int D>
struct DqGemmCfg {
  static constexpr int kStages = 3;
  static constexpr int kThreads = 192;
  static constexpr int kTileBytes = 128 * D;  // one Kt tile
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  // TMEM: dQ accumulator [0, D), then dS and K scale slots, 4 columns per
  // pipeline stage
  static constexpr uint32_t kColDQ = 0, kSfDS = D /*+4s*/, kSfKt = D + 16 /*+4s*/;
  static constexpr uint32_t kTmemCols = D == 128 ? 256 : 128;
  // shared memory per stage: dS tile (16 KB), Kt tile, Kt atom, 16 dS block
  // scales (padded so stages stay 1024-byte aligned)
  static constexpr int kOffKt = 16384, kOffKtSf = 16384 + kTileBytes, kOffDsSf = kOffKtSf + kAtomBytes;
  static constexpr int kStageBytes = 16384 + kTileBytes + 1024;
  static constexpr int kOffSfOne = kStages * kStageBytes;       // a scale-1 atom (strict dQ's diagonal K)
  static constexpr int kSmemBytes = kOffSfOne + kAtomBytes + 1024;
};

}  // namespace

template <int D, bool F16, bool STRICT>
__global__ void __launch_bounds__(DqGemmCfg<D>::kThreads, 2)
    attn_dq_gemm_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = DqGemmCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_full[C::kStages], bar_empty[C::kStages], bar_sfa[C::kStages], bar_final, bar_drain,
      bar_pfull, bar_pfree;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot;

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
  if (ktile_base < 0) ktile_base = doc_tile_base(a.cu_k, b, nk, tid, C::kThreads, &s_slot);

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
      mbar_init(&bar_sfa[s], 128);  // the four epilogue warps
    }
    mbar_init(&bar_final, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_pfull, 1);
    mbar_init(&bar_pfree, 128);  // the four epilogue warps
    s_abort = 0;
    fence_barrier_init();
  }
  if constexpr (STRICT) {
    for (int i = tid; i < kAtomBytes / 16; i += C::kThreads)
      reinterpret_cast<uint4*>(smem + C::kOffSfOne)[i] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages &&
            !role_wait(&bar_empty[s], ((j / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma))
          break;
        // pair (h, b, key tile j, query tile qt)
        const int64_t pair = (static_cast<int64_t>(h) * a.ntiles_k + ktile_base + j) * a.mt + qt;
        const int k0 = static_cast<int>(kdoc_start + static_cast<int64_t>(j) * 128);
        const int64_t katom = (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + j) * kAtomBytes;
        uint8_t* st = smem + s * C::kStageBytes;
        // strict dQ: one scale per (query row, 32 keys) -- a whole atom per
        // pair -- and the per-key K codes on the diagonal pair
        const bool kdiag = STRICT && a.causal && j == qt;
        mbar_arrive_expect_tx(&bar_full[s], 16384 + C::kTileBytes + kAtomBytes + (STRICT ? kAtomBytes : 16));
        bulk_load(st, a.ds_codes + pair * 16384, 16384, &bar_full[s]);  // stored as its swizzled image
        tma_load_3d(st + C::kOffKt, kdiag ? &maps.kkey : &maps.kt, &bar_full[s], 0, hk, k0);
        bulk_load(st + C::kOffKtSf, a.kt_sf + katom, kAtomBytes, &bar_full[s]);
        if constexpr (STRICT) bulk_load(st + C::kOffDsSf, a.ds_sf + pair * kAtomBytes, kAtomBytes, &bar_full[s]);
        else bulk_load(st + C::kOffDsSf, a.ds_sf + pair * 16, 16, &bar_full[s]);
        issued = j + 1;
      }
      for (int j = (issued > C::kStages ? issued - C::kStages : 0); j < issued; ++j)
        mbar_wait(&bar_full[j % C::kStages], (j / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint64_t dA0 = make_sdesc(smem_u32(smem), 16, 1024, kSwz128);           // dS: 128-byte query rows
      const uint64_t dB0 = make_sdesc(smem_u32(smem + C::kOffKt), 16, C::kSBO, C::kSwz);  // Kt
      const uint64_t dSf0 = atom_desc(smem + C::kOffKtSf);
      bool ok = true;
      for (int j = 0; j < n_kt; ++j) {
        const int s = j % C::kStages;
        // operands landed and the epilogue warps have laid out the dS scales
        if (!(ok = role_wait(&bar_full[s], (j / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (!(ok = role_wait(&bar_sfa[s], (j / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        // F16: the previous partial must have been read out of TMEM
        if (F16 && j > 0 && !(ok = role_wait(&bar_pfree, (j - 1) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        const uint32_t tSfA = tmem + C::kSfDS + 4 * s, tSfB = tmem + C::kSfKt + 4 * s;
        tmem_cp_desc(tSfB, (STRICT && a.causal && j == qt) ? atom_desc(smem + C::kOffSfOne)
                                                           : sdesc_adv(dSf0, s * C::kStageBytes));
        const uint64_t da = sdesc_adv(dA0, s * C::kStageBytes), db = sdesc_adv(dB0, s * C::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 32 keys per step: 32 rows of each operand
          mma_mxf8_ss(tmem + C::kColDQ, sdesc_adv(da, kk * 4096), sdesc_adv(db, kk * 32 * D),
                      make_idesc_mxf8(128, D, 1, 1, kk, kk), tSfA, tSfB, ((!F16 && j > 0) || kk > 0) ? 1u : 0u);
        mma_commit(&bar_empty[s]);
        if (F16) mma_commit(&bar_pfull);
      }
      mma_commit(&bar_final);
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int64_t qpos = static_cast<int64_t>(qt) * 128 + r;
    // per key tile: the scales of this warp's 32 query rows (query block
    // `quad`) for the 4 key blocks go to lane r, column kSfDS + 4 s + r / 32,
    // byte = key block -- the A scale-factor layout of the MMA.  Stage s was
    // reloaded only after the MMAs of tile j - kStages completed, so its
    // slot is free.
    bool ok = true;
    // F16: this row's fp16 sum, two channels per register
    __half2 acc[F16 ? D / 2 : 1];
    if constexpr (F16) {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) acc[i] = __float2half2_rn(0.0f);
    }
    // alpha and the boost of the fp16 sum: 2^9, or the row's own 2^beta
    float boost = 512.0f;
    if (F16 && a.dq_boost != nullptr && qpos < n) boost = a.dq_boost[static_cast<int64_t>(h) * a.T + doc_start + qpos];
    const float bst = a.alpha * boost;
    const float unboost = __uint_as_float((254u << 23) - __float_as_uint(boost));  // 2^-beta, exact
    // fold the partial of key tile jj into the fp16 sum (F16 only)
    auto fold = [&](int jj) -> bool {
      if (!warp_wait(&bar_pfull, jj & 1, abort_flag, a.err, kErrTimeoutEpilogue)) return false;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::kColDQ + c, rr);
        tmem_ld_wait();
        if (c + 32 == D) {  // every column read: tile jj + 1 may overwrite them
          tc_fence_before();
          mbar_arrive(&bar_pfree);
        }
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          acc[(c + i) / 2] = __hadd2(acc[(c + i) / 2], __floats2half2_rn(__uint_as_float(rr[i]) * bst,
                                                                           __uint_as_float(rr[i + 1]) * bst));
      }
      return true;
    };
    for (int j = 0; j < n_kt; ++j) {
      const int s = j % C::kStages;
      if (!(ok = warp_wait(&bar_full[s], (j / C::kStages) & 1, abort_flag, a.err, kErrTimeoutEpilogue))) break;
      // default: the 16 block scales, one word per query block; strict: the
      // atom's word of this lane's query row (byte = key block)
      const uint32_t sc = *reinterpret_cast<const uint32_t*>(smem + s * C::kStageBytes + C::kOffDsSf +
                                                             (STRICT ? lane * 16 + quad * 4 : 4 * quad));
      tmem_st1(lane_base + C::kSfDS + 4 * s + quad, sc);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_sfa[s]);
      if constexpr (F16) {
        if (j > 0 && !(ok = fold(j - 1))) break;
      }
    }
    if constexpr (F16) {
      if (ok && n_kt > 0) ok = fold(n_kt - 1);
    }
    if (ok) ok = role_wait(&bar_final, 0, abort_flag, a.err, kErrTimeoutEpilogue);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int64_t t = doc_start + qpos;
      __nv_bfloat16* dqrow = reinterpret_cast<__nv_bfloat16*>(a.dq_out) + (t * a.Hq + h) * D;
      if constexpr (F16) {
        if (qpos < n) {
#pragma unroll
          for (int c = 0; c < D; c += 8) {
            uint4 v;
            uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = __half22float2(acc[c / 2 + k]);
              vw[k] = pack_bf16x2(f.x * unboost, f.y * unboost);
            }
            *reinterpret_cast<uint4*>(dqrow + c) = v;
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t rr[32];
          tmem_ld32(lane_base + C::kColDQ + c, rr);
          tmem_ld_wait();
          if (qpos < n) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(rr[i]) * a.alpha, __uint_as_float(rr[i + 1]) * a.alpha);
              v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * a.alpha, __uint_as_float(rr[i + 3]) * a.alpha);
              v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * a.alpha, __uint_as_float(rr[i + 5]) * a.alpha);
              v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * a.alpha, __uint_as_float(rr[i + 7]) * a.alpha);
              *reinterpret_cast<uint4*>(dqrow + c + i) = v;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

namespace {

template <int D, bool F16, bool STRICT>
cudaError_t launch_dq_gemm_t(const BwdArgs& a, const BwdMaps& m, int max_seqlen, cudaStream_t stream) {
  using C = DqGemmCfg<D>;
  const dim3 grid = a.q_items ? dim3(static_cast<unsigned>(a.ntiles * a.Hq))
                              : dim3((max_seqlen + 127) / 128, a.num_docs, a.Hq);
  cudaError_t e = cudaFuncSetAttribute(attn_dq_gemm_kernel<D, F16, STRICT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_dq_gemm_kernel<D, F16, STRICT><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_gemm_d(const BwdArgs& a, const BwdMaps& m, int max_seqlen, cudaStream_t stream) {
  const bool f16 = a.dq_mode != 0;  // FP16 x 2^9 or the per-row boost
  if (a.kkey_sf != nullptr)
    return f16 ? launch_dq_gemm_t<D, true, true>(a, m, max_seqlen, stream)
               : launch_dq_gemm_t<D, false, true>(a, m, max_seqlen, stream);
  return f16 ? launch_dq_gemm_t<D, true, false>(a, m, max_seqlen, stream)
             : launch_dq_gemm_t<D, false, false>(a, m, max_seqlen, stream);
}

}  // namespace

cudaError_t launch_dq_gemm(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  return d == 128 ? launch_dq_gemm_d<128>(a, m, max_seqlen, stream) : launch_dq_gemm_d<64>(a, m, max_seqlen, stream);
}

}  // namespace mxa
