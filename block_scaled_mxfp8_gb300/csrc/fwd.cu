// fwd.cu -- MXFP8 block-scaled attention forward (tcgen05, TMEM, TMA).
//
// A CTA computes 128-query tiles of (document, query head) items one after
// another (persistent launches: each running CTA takes over the items of
// CTAs not yet started), walking each tile's visible keys 256 at a time:
//   S_j  = Q K_j^T          block-scaled MXFP8 MMA (kind::mxf8f6f4), M = 128
//                           queries, N = 256 keys (per key, half the MMA
//                           groups, barrier round trips and pipe drains of
//                           N = 128; a double-buffered N = 128 variant
//                           measured 1.36x slower), Q/K ROW-view scales in
//                           TMEM;
//   P_j  = online softmax of alpha * S_j with a lazily updated row max
//          (rescale only when the tile max exceeds the running max by more
//          than tau = 4 in log2 units; the reference is ceil of the max, an
//          integer in log2 units), quantized in registers as E4M3(2^4 p)
//          (FLAMIA notes sec. 5: 2^(c+tau) <= 448 with (c, tau) = (4, 4)),
//          stored to TMEM;
//   [O | L] += P_j [V_j | 1]  one block-scaled MMA with A = P from TMEM
//          (scale 2^(m - mo - 4): O and L keep a reference mo up to 32
//          binades behind the row max m, so that a raise of m rescales
//          nothing in TMEM; the strict mode keeps mo = m) and B = V
//          (MN-major, TOK-view scales) widened by 16
//          columns of ones, so that L is the row sum of exactly the quantized
//          weights used for O (the ones come from one shared 4 KB block that
//          every K step reaches through the descriptor's leading byte offset);
//   O = O / L -> bf16, LSE = m + ln l with l the fp32 sum of the unquantized
//   weights (FLAMIA notes sec. 2, online softmax).
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM owner and S issuer,
// warp 18 = P V issuer (an MMA issue blocks its thread for about the pipe
// time, so S_{j+1} must not queue behind P_{j-1} V), warps 2..17 = softmax /
// correction / epilogue: four warps per TMEM lane
// quadrant, each taking 64 of the 256 key columns of its 32 query rows.  A
// softmax warp copies its S columns into registers and releases S at once,
// so the next S MMA runs while the exponentials of this tile are formed; the
// four warps of a quadrant merge their row maxima through shared memory.
// K and V tiles stream through separate three-stage rings (256 keys per
// stage).
//
// Strict causal mode (a per-key view of V given): on each query's diagonal
// 128-key tile, where a 32-key scale group of V would straddle the query,
// every key carries its own power-of-two scale 2^e_k, folded into the
// probability operand (FLAMIA notes sec. 4): P'_ik = p_ik 2^e_k is
// quantized per query row and 32 keys by the MX rule, multiplied with the
// per-key codes (B scale 1), and the MMA of those K steps runs with N = D so
// that the ones column skips them; the weights the codes stand for,
// q(P') 2^e_blk 2^-e_k, are summed in registers and added to L at the end.
//
// TMEM columns: S [0,256), O [256,256+D) and L [256+D,256+D+16), Q-scale 400,
// K-scale 404 + 8 (j mod 2) (two atoms per 256 keys), V-scale atoms 420 and 428 each
// followed by a column block of 1.0 for the ones rows, P-scale 436, the folded
// P' scales 440 (K steps 0, 1 of the diagonal half) and 444 (K steps 2, 3), P
// [448,512).
#include <cuda_bf16.h>

#include "attn_common.cuh"

namespace mxa {

namespace {

template <int D>
struct FwdCfg {
  static constexpr int kStages = 3;
  static constexpr int kHalfBytes = 128 * D;          // one 128-key box of K or V
  static constexpr int kKVBytes = 2 * kHalfBytes;     // 256 keys
  static constexpr uint32_t kSwz = D == 128 ? kSwz128 : kSwz64;
  static constexpr uint32_t kSBO = 8 * D;
  static constexpr int kKSteps = D / 32;              // K steps of S = Q K^T
  static constexpr int kKStepBytes = 32 * D;          // 32 keys of V (P V K step)
  static constexpr int kThreads = 608;                // 3 role warps + 16 softmax warps
  static constexpr int kSoftmaxThreads = 512;
  static constexpr uint32_t kColS = 0, kColO = 256, kColL = 256 + D, kColSfQ = 400, kColSfK = 404, kColSfVA = 420,
                            kColOneA = 424, kColSfVB = 428, kColOneB = 432, kColSfP = 436, kColSfPd = 440,
                            kColP = 448;
  // shared memory map (offsets from the 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 128 * D;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffOnes = kOffV + kStages * kKVBytes;  // 32 rows x D bytes of E4M3 1.0
  static constexpr int kOffSfQ = kOffOnes + 4096;
  static constexpr int kOffSfK = kOffSfQ + kAtomBytes;         // 2 atoms per stage
  static constexpr int kOffSfV = kOffSfK + kStages * 2 * kAtomBytes;
  static constexpr int kOffSfOne = kOffSfV + kStages * 2 * kAtomBytes;  // an atom of scale 1.0 (per-key V codes)
  static constexpr int kSmemBytes = kOffSfOne + kAtomBytes + 1024;      // + alignment slack
};

// Row maximum of 64 scores in four independent chains.
__device__ __forceinline__ float max64(const float (&v)[64]) {
  float a = fmax3(v[0], v[1], v[2]), b = fmax3(v[3], v[4], v[5]), c = fmax3(v[6], v[7], v[8]),
        d = fmax3(v[9], v[10], v[11]);
#pragma unroll
  for (int i = 12; i < 60; i += 8) {
    a = fmax3(a, v[i], v[i + 1]);
    b = fmax3(b, v[i + 2], v[i + 3]);
    c = fmax3(c, v[i + 4], v[i + 5]);
    d = fmax3(d, v[i + 6], v[i + 7]);
  }
  a = fmax3(a, v[60], v[61]);
  b = fmax3(b, v[62], v[63]);
  return fmax3(fmaxf(a, b), c, d);
}

__device__ __forceinline__ void ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t x0[32], x1[32];
  tmem_ld32(taddr, x0);
  tmem_ld32(taddr + 32, x1);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(x0[i]);
    v[32 + i] = __uint_as_float(x1[i]);
  }
}

// 64 fp32 columns and their maximum, from the loads themselves (the TMEM read
// merged with the row-max reduction, FLAMIA notes sec. 7) -- for key tiles
// whose columns are all visible.
__device__ __forceinline__ void ld64_max(uint32_t taddr, float (&v)[64], float& mx) {
  float m0, m1;
  tmem_ld32_max(taddr, *reinterpret_cast<float(*)[32]>(&v[0]), m0);
  tmem_ld32_max(taddr + 32, *reinterpret_cast<float(*)[32]>(&v[32]), m1);
  tmem_ld_wait();
  mx = fmaxf(m0, m1);
}

// Most binades by which O and L may trail the P reference m in the default
// mode (each of their weights then reaches 2^(kOLag + 4): fp32 headroom for
// |V| up to ~2^70 at hundreds of thousands of keys).  The strict mode keeps
// them on m, as its diagonal fold scales are formed against m.
constexpr float kOLag = 32.0f;

// 2^(b - 127) of a UE8M0 byte (b = 0: 2^-127).
__device__ __forceinline__ float ue8m0_f32(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// The diagonal tile's fold for one thread's 64 key columns, 32 at a time,
// read again from TMEM at tS (the warps release S only after this read):
// the weights p = 2^(s sl2 - m + 4) (summed into lsa/lsb as elsewhere),
// times 2^e_k of each key (kexp: its 64 exponent bytes, 16-byte aligned),
// quantized per 32 keys by the MX rule into pw; columns at or past lim are
// masked.  The block's MMA scale is 2^(e_blk - 4), which also removes the
// boost.  Returns the sum of the weights the codes stand for,
// code 2^(e_blk - 4) 2^-e_k (the units of the L column); the two block scale
// bytes go to sfb (byte blk).
// Out of line: it runs once per CTA, and kept apart its temporaries do not
// raise the register demand of the main loop.
struct FoldOut {
  uint32_t pw[16];
  uint32_t sfb;
  float lw;
  uint64_t lsa, lsb;
};

__device__ __noinline__ FoldOut fold_keys(uint32_t tS, int col0, int lim, const uint8_t* kexp, uint64_t sl2x2,
                                          uint64_t neg2, uint64_t lsa, uint64_t lsb) {
  FoldOut out;
  uint32_t (&pw)[16] = out.pw;
  uint32_t& sfb = out.sfb;
  float lw = 0.0f;
  sfb = 0u;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float x[32];
    {
      uint32_t rr[32];
      tmem_ld32(tS + 32 * blk, rr);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) x[c] = (col0 + 32 * blk + c < lim) ? __uint_as_float(rr[c]) : -INFINITY;
    }
    float am = 0.0f;
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const float2 x01 = f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sl2x2, neg2));
      const float2 x23 = f2_unpack(f2_fma(f2_pack(x[c + 2], x[c + 3]), sl2x2, neg2));
      const float p0 = ex2_approx(x01.x), p1 = ex2_approx(x01.y);
      const float p2 = ex2_approx(x23.x), p3 = ex2_approx(x23.y);
      lsa = f2_add(lsa, f2_pack(p0, p1));
      lsb = f2_add(lsb, f2_pack(p2, p3));
      const uint32_t eb = __ldg(reinterpret_cast<const uint32_t*>(kexp + 32 * blk + c));
      x[c] = p0 * ue8m0_f32(eb & 0xFFu);
      x[c + 1] = p1 * ue8m0_f32((eb >> 8) & 0xFFu);
      x[c + 2] = p2 * ue8m0_f32((eb >> 16) & 0xFFu);
      x[c + 3] = p3 * ue8m0_f32(eb >> 24);
      am = fmax3(am, fmaxf(x[c], x[c + 1]), fmaxf(x[c + 2], x[c + 3]));
    }
    const int e = mx_exponent_bits(__float_as_uint(am));
    const float sc = exp2i_neg(e);
    // the block's MMA scale 2^(e - 4) also takes out the 2^4 boost that p
    // carries (the other K steps' constant 2^-4)
    const int sb = e + 127 - 4 < 0 ? 0 : e + 127 - 4;
    const float up = ue8m0_f32(static_cast<uint32_t>(sb));
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const uint32_t w = pack_e4m3x4(x[c] * sc, x[c + 1] * sc, x[c + 2] * sc, x[c + 3] * sc);
      pw[8 * blk + (c >> 2)] = w;
      const float2 d01 = e4m3x2_to_f32x2(w & 0xFFFFu), d23 = e4m3x2_to_f32x2(w >> 16);
      const uint32_t eb = __ldg(reinterpret_cast<const uint32_t*>(kexp + 32 * blk + c));
      lw += (d01.x * up) * exp2i_neg(static_cast<int>(eb & 0xFFu) - 127);
      lw += (d01.y * up) * exp2i_neg(static_cast<int>((eb >> 8) & 0xFFu) - 127);
      lw += (d23.x * up) * exp2i_neg(static_cast<int>((eb >> 16) & 0xFFu) - 127);
      lw += (d23.y * up) * exp2i_neg(static_cast<int>(eb >> 24) - 127);
    }
    sfb |= static_cast<uint32_t>(sb) << (8 * blk);
  }
  out.lw = lw;
  out.lsa = lsa;
  out.lsb = lsb;
  return out;
}

// One forward work item: a (document, 128-query tile, query head) and the
// document's first scale tiles on the query and key sides.
struct FwdItem {
  int b, h, qt;
  int64_t tile_base, ktile_base;
};

// Item v of a persistent launch: item v / Hq of the cost-sorted list for head
// v % Hq, or the v-th (query tile, document, head) of equal documents --
// query tiles fastest, so the CTAs running together share a head's K and V
// tiles in L2, heaviest first when causal, and the last groups' query tiles
// interleaved heaviest first (causal_launch_order).  False past the last
// item.
__device__ __forceinline__ bool fwd_item(const FwdArgs& a, int64_t v, FwdItem& it) {
  if (a.items) {
    const int64_t i = v / a.Hq;
    if (i >= __ldg(a.item_count)) return false;
    it.h = static_cast<int>(v - i * a.Hq);
    const int4 e = __ldg(reinterpret_cast<const int4*>(a.items + i));
    it.b = e.x;
    it.qt = e.y;
    it.tile_base = e.z;
    it.ktile_base = e.w;
    return true;
  }
  const int nqt = a.nq_tiles_doc;
  if (v >= static_cast<int64_t>(nqt) * a.num_docs * a.Hq) return false;
  if (a.causal) {
    int grp, qi;
    causal_launch_order(static_cast<int>(v), a.num_docs * a.Hq, nqt, grp, qi);
    it.b = grp % a.num_docs;
    it.h = grp / a.num_docs;
    it.qt = nqt - 1 - qi;
  } else {
    const int qi = static_cast<int>(v % nqt);
    const int64_t rest = v / nqt;
    it.b = static_cast<int>(rest % a.num_docs);
    it.h = static_cast<int>(rest / a.num_docs);
    it.qt = qi;
  }
  it.tile_base = static_cast<int64_t>(it.b) * nqt;
  it.ktile_base = static_cast<int64_t>(it.b) * a.nk_tiles_doc;
  return true;
}

// Geometry of one item.
struct FwdGeo {
  int hk, nk_tiles, n_it, dh;
  int64_t doc_start, n, kdoc_start, nk;
};
__device__ __forceinline__ FwdGeo fwd_geo(const FwdArgs& a, const FwdItem& it) {
  FwdGeo g;
  g.hk = it.h / (a.Hq / a.Hkv);
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, it.b, g.doc_start, g.n);
  doc_bounds(a.cu_k, a.num_docs, a.Tk, it.b, g.kdoc_start, g.nk);
  g.nk_tiles = static_cast<int>((g.nk + 127) / 128);
  // visible keys [0, nkeys), walked 256 at a time
  const int64_t nkeys = a.causal ? min(g.nk, static_cast<int64_t>(it.qt + 1) * 128) : g.nk;
  g.n_it = static_cast<int>((nkeys + 255) / 256);
  g.dh = it.qt & 1;  // strict causal fold: the last iteration's half (qt % 2) is the diagonal tile
  return g;
}

}  // namespace

template <int D, bool FOLD, bool PERSIST>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ uint64_t bar_q, bar_q_free, bar_k_full[C::kStages], bar_k_empty[C::kStages], bar_v_full[C::kStages],
      bar_v_empty[C::kStages], bar_s_full, bar_s_empty, bar_p_full, bar_o_done, bar_o_free, bar_drain, bar_drain2,
      bar_mx[2][4], bar_lsum, bar_clc[2], bar_clc_free[2];
  __shared__ alignas(16) uint4 s_clc[2];  // cluster-launch-control responses, by item parity
  __shared__ float s_mx[2][4][128];  // [iteration parity][column quarter][row] partial row maxima
  __shared__ float s_l[4][128];      // [column quarter][row] partial row sums
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int64_t s_slot, s_slot_k;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The CTA's items.  Persistent launches (a cost-sorted list, or equal
  // documents) start with item blockIdx.x of a grid with one CTA per item,
  // heaviest first, and then take over the items of CTAs that have not
  // started yet (cluster launch control): the producer asks for one after
  // the last K/V load of each item, and every role reads the answer at the
  // end of that item -- all roles walk the same sequence, with each
  // barrier's phase counted across items.  Packed documents without a list
  // take one item per CTA from the max_seqlen grid (heaviest query tiles
  // first when causal).
  FwdItem item0;
  if constexpr (PERSIST) {
    if (!fwd_item(a, blockIdx.x, item0)) return;
  } else {
    item0.b = blockIdx.y;
    item0.h = blockIdx.z;
    item0.qt = a.causal ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
    int64_t ds, dn, ks, kn;
    doc_bounds(a.cu_seqlens, a.num_docs, a.T, item0.b, ds, dn);
    doc_bounds(a.cu_k, a.num_docs, a.Tk, item0.b, ks, kn);
    if (item0.qt >= static_cast<int>((dn + 127) / 128)) return;
    item0.tile_base = doc_tile_base(a.cu_seqlens, item0.b, dn, tid, C::kThreads, &s_slot);
    item0.ktile_base = (a.cu_k == a.cu_seqlens && a.Tk == a.T)
                           ? item0.tile_base
                           : doc_tile_base(a.cu_k, item0.b, kn, tid, C::kThreads, &s_slot_k);
  }
  // The item after the CTA's n-th (false at the end of the sequence, or when
  // the wait fails): the response in slot n & 1, read once its phase is
  // complete; `release` arrives on the slot's free barrier (one thread per
  // role and one lane per softmax warp).
  auto next_item = [&](int n, FwdItem& it, bool release, bool& ok) -> bool {
    if constexpr (!PERSIST) {
      return false;
    } else {
      const bool got = role_wait(&bar_clc[n & 1], (n >> 1) & 1, &s_abort, a.err, kErrTimeoutOther);
      uint32_t x = 0;
      const bool more = got && clc_query(&s_clc[n & 1], x);
      if (release) mbar_arrive(&bar_clc_free[n & 1]);
      if (!got) ok = false;
      return more && fwd_item(a, x, it);
    }
  };

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_q_free, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_v_empty[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_s_empty, C::kSoftmaxThreads);
    mbar_init(&bar_p_full, C::kSoftmaxThreads);
    mbar_init(&bar_o_done, 1);
    mbar_init(&bar_o_free, C::kSoftmaxThreads);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_drain2, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&bar_mx[0][q], 128);
      mbar_init(&bar_mx[1][q], 128);
    }
    mbar_init(&bar_lsum, C::kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_clc[i], 1);
      mbar_init(&bar_clc_free[i], 3 + C::kSoftmaxThreads / 32);  // producer, two MMA issuers, softmax warps
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  for (int i = tid; i < 4096 / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kOffOnes)[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
  for (int i = tid; i < kAtomBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kOffSfOne)[i] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const bool fold = FOLD && a.causal;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      // K and V stream through separate rings: a K stage is released as soon
      // as its S MMA has completed, a V stage after its P V MMA, so the keys
      // of later tiles -- and of the next item -- are loaded well ahead of
      // the P V chain.  The next item's Q loads once the S MMAs of the
      // previous item are done with Q.
      uint32_t issued_k = 0, issued_v = 0;  // ring iterations, counted across items
      int issued_q = 0;
      bool ok = true;
      FwdItem itm = item0;
      int n = 0;  // items of this CTA so far
      do {
        const FwdGeo G = fwd_geo(a, itm);
        const int hk = G.hk, h = itm.h, qt = itm.qt, n_it = G.n_it, dh = G.dh, nk_tiles = G.nk_tiles;
        const int64_t kdoc_start = G.kdoc_start, ktile_base = itm.ktile_base;
        if (issued_q >= 1 &&
            !(ok = role_wait(&bar_q_free, (issued_q - 1) & 1, abort_flag, a.err, kErrTimeoutTma)))
          break;
        const int q0 = static_cast<int>(G.doc_start + static_cast<int64_t>(qt) * 128);
        mbar_arrive_expect_tx(&bar_q, 128 * D + kAtomBytes);
        tma_load_3d(smem + C::kOffQ, &maps.q, &bar_q, 0, h, q0);
        bulk_load(smem + C::kOffSfQ,
                  a.q_sf + ((static_cast<int64_t>(h) * a.ntiles + itm.tile_base + qt) * kAtomBytes), kAtomBytes,
                  &bar_q);
        ++issued_q;
        for (int j = 0; ok && j < n_it; ++j) {
        const uint32_t gk = issued_k;
        const int s = static_cast<int>(gk % C::kStages);
        const int t0 = 2 * j;  // first 128-key tile of this iteration
        // the second half may lie past the document: reuse the first half's
        // atoms then (its keys are masked; the scales just have to be finite)
        const int t1 = (t0 + 1 < nk_tiles) ? t0 + 1 : t0;
        const int k0 = static_cast<int>(kdoc_start + static_cast<int64_t>(t0) * 128);
        const int64_t atom0 = (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + t0) * kAtomBytes;
        const int64_t atom1 = (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + t1) * kAtomBytes;
        if (gk >= C::kStages &&
            !(ok = role_wait(&bar_k_empty[s], ((gk / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma)))
          break;
        uint8_t* sk = smem + C::kOffK + s * C::kKVBytes;
        uint8_t* sfk = smem + C::kOffSfK + s * 2 * kAtomBytes;
        mbar_arrive_expect_tx(&bar_k_full[s], C::kKVBytes + 2 * kAtomBytes);
        tma_load_3d(sk, &maps.k, &bar_k_full[s], 0, hk, k0);
        tma_load_3d(sk + C::kHalfBytes, &maps.k, &bar_k_full[s], 0, hk, k0 + 128);
        bulk_load(sfk, a.k_sf + atom0, kAtomBytes, &bar_k_full[s]);
        bulk_load(sfk + kAtomBytes, a.k_sf + atom1, kAtomBytes, &bar_k_full[s]);
        issued_k = gk + 1;
        if (gk >= C::kStages &&
            !(ok = role_wait(&bar_v_empty[s], ((gk / C::kStages) - 1) & 1, abort_flag, a.err, kErrTimeoutTma)))
          break;
        uint8_t* sv = smem + C::kOffV + s * C::kKVBytes;
        uint8_t* sfv = smem + C::kOffSfV + s * 2 * kAtomBytes;
        mbar_arrive_expect_tx(&bar_v_full[s], C::kKVBytes + 2 * kAtomBytes);
        const bool fold_it = fold && j == n_it - 1;  // the diagonal half from the per-key view
        tma_load_3d(sv, (fold_it && dh == 0) ? &maps.vkey : &maps.v, &bar_v_full[s], 0, hk, k0);
        tma_load_3d(sv + C::kHalfBytes, (fold_it && dh == 1) ? &maps.vkey : &maps.v, &bar_v_full[s], 0, hk, k0 + 128);
        bulk_load(sfv, a.v_sf + atom0, kAtomBytes, &bar_v_full[s]);
        bulk_load(sfv + kAtomBytes, a.v_sf + atom1, kAtomBytes, &bar_v_full[s]);
        issued_v = gk + 1;
        }
        if (!ok) break;
        if constexpr (PERSIST) {
          // dynamic fetch after the item's last K/V load: the slot is free
          // once every role has read the response of item n - 2
          if (n >= 2 && !(ok = role_wait(&bar_clc_free[n & 1], ((n >> 1) - 1) & 1, abort_flag, a.err,
                                         kErrTimeoutOther)))
            break;
          clc_try_cancel(&s_clc[n & 1], &bar_clc[n & 1]);
        }
      } while (next_item(n++, itm, true, ok) && ok);
      // drain: every load issued must have landed before the CTA exits
      if (issued_q) role_wait(&bar_q, (issued_q - 1) & 1, abort_flag, nullptr, 0);
      for (uint32_t j = (issued_k > C::kStages ? issued_k - C::kStages : 0); j < issued_k; ++j)
        mbar_wait(&bar_k_full[j % C::kStages], (j / C::kStages) & 1, nullptr, 0);
      for (uint32_t j = (issued_v > C::kStages ? issued_v - C::kStages : 0); j < issued_v; ++j)
        mbar_wait(&bar_v_full[j % C::kStages], (j / C::kStages) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      // descriptors built once; per MMA only constant offsets are added
      const uint64_t dQa = make_sdesc(smem_u32(smem + C::kOffQ), 16, C::kSBO, C::kSwz);
      const uint64_t dK0 = make_sdesc(smem_u32(smem + C::kOffK), 16, C::kSBO, C::kSwz);
      const uint64_t dSfK0 = atom_desc(smem + C::kOffSfK);
      const uint32_t tS = tmem + C::kColS, tSfQ = tmem + C::kColSfQ;
      bool ok = true;
      // S = Q K^T, 128 x 256, for ring iteration g (j: its index in the item)
      auto issue_s = [&](uint32_t g, int j) -> bool {
        const int s = static_cast<int>(g % C::kStages);
        if (!role_wait(&bar_k_full[s], (g / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        if (g >= 1 && !role_wait(&bar_s_empty, (g - 1) & 1, abort_flag, a.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        // the item's Q scales, once the previous S MMA (which read the
        // previous item's) has completed and been read out
        if (j == 0) tmem_cp_atom(tSfQ, smem + C::kOffSfQ);
        // K-scale slots alternate between two pairs of atoms (an S MMA may be
        // issued while the previous one is still in the pipe)
        const uint32_t tSfK = tmem + C::kColSfK + 8 * static_cast<uint32_t>(g & 1);
        const uint64_t dsf = sdesc_adv(dSfK0, s * 2 * kAtomBytes);
        tmem_cp_desc(tSfK, dsf);
        tmem_cp_desc(tSfK + 4, sdesc_adv(dsf, kAtomBytes));
        const uint64_t dk = sdesc_adv(dK0, s * C::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk)
          mma_mxf8_ss(tS, sdesc_adv(dQa, 32 * kk), sdesc_adv(dk, 32 * kk), make_idesc_mxf8(128, 256, 0, 0, kk, kk),
                      tSfQ, tSfK, kk > 0);
        mma_commit(&bar_s_full);
        mma_commit(&bar_k_empty[s]);
        return true;
      };
      uint32_t g = 0;
      int n_items = 0;
      FwdItem itm = item0;
      do {
        const int n_it = fwd_geo(a, itm).n_it;
        if (!(ok = role_wait(&bar_q, n_items & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        for (int j = 0; ok && j < n_it; ++j, ++g)
          if (!(ok = issue_s(g, j))) break;  // waits until S_{g-1} has been read out
        if (!ok) break;
        mma_commit(&bar_q_free);  // this item's S MMAs are done with Q once they complete
      } while (next_item(n_items++, itm, true, ok) && ok);
      // drain this thread's MMAs before the TMEM is released
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, 0);
    }
  } else if (warp == 18) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      // the P V operand B = [V | 1] keeps its second atom column (the ones
      // block) fixed, so stepping its start address by x bytes lowers its
      // leading byte offset by x
      const uint32_t onesa = smem_u32(smem + C::kOffOnes), va0 = smem_u32(smem + C::kOffV);
      const uint64_t dV0 = make_sdesc(va0, onesa - va0, C::kSBO, C::kSwz);
      const uint64_t dSfV0 = atom_desc(smem + C::kOffSfV);
      auto v_adv = [](uint64_t d, uint32_t bytes) -> uint64_t {
        return d + (bytes >> 4) - (static_cast<uint64_t>(bytes >> 4) << 16);
      };
      const uint32_t tO = tmem + C::kColO, tP = tmem + C::kColP, tSfP = tmem + C::kColSfP, tSfPd = tmem + C::kColSfPd;
      const uint64_t dSfOne = atom_desc(smem + C::kOffSfOne);
      const uint32_t tSfVA = tmem + C::kColSfVA, tSfVB = tmem + C::kColSfVB;
      // The first P V MMA of an item restarts [O | L]; the softmax warps
      // arrive on p_full for an item only after all of them have read the
      // previous item's O and L (bar_o_free), so waiting for p_full orders it.
      uint32_t g = 0;
      bool ok = true;
      FwdItem itm = item0;
      int n = 0;
      do {
      const FwdGeo G = fwd_geo(a, itm);
      const int n_it = G.n_it, dh = G.dh;
      for (int j = 0; j < n_it; ++j, ++g) {
        const int s = static_cast<int>(g % C::kStages);
        if (!(ok = role_wait(&bar_v_full[s], (g / C::kStages) & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        if (!(ok = role_wait(&bar_p_full, g & 1, abort_flag, a.err, kErrTimeoutMma))) break;
        tc_fence_after();
        const bool fold_it = fold && j == n_it - 1;
        const uint64_t dsf = sdesc_adv(dSfV0, s * 2 * kAtomBytes);
        tmem_cp_desc(tSfVA, (fold_it && dh == 0) ? dSfOne : dsf);
        tmem_cp_desc(tSfVB, (fold_it && dh == 1) ? dSfOne : sdesc_adv(dsf, kAtomBytes));
        const uint64_t dv = v_adv(dV0, s * C::kKVBytes);
        // the folded half goes last, so that the first K step of the first
        // iteration -- the one that starts the sums -- also writes L
        const int rot = (fold_it && dh == 0) ? 4 : 0;
#pragma unroll
        for (int ki = 0; ki < 8; ++ki) {  // [O | L] += P [V | 1], 32 keys per step
          const int kk = (ki + rot) & 7;
          // folded K steps: per-row P' scales, per-key codes, and N = D (L is summed in registers)
          const bool fk = fold_it && (kk >> 2) == dh;
          mma_mxf8_ts(tO, tP + 8 * kk, v_adv(dv, kk * C::kKStepBytes),
                      make_idesc_mxf8(128, fk ? D : D + 16, 0, 1, kk & 3, kk & 3),
                      fk ? tSfPd + ((kk & 2) ? 4u : 0u) : tSfP, kk < 4 ? tSfVA : tSfVB, (j > 0 || ki > 0) ? 1u : 0u);
        }
        mma_commit(&bar_o_done);
        mma_commit(&bar_v_empty[s]);
      }
      if (!ok) break;
      } while (next_item(n++, itm, true, ok) && ok);
      mma_commit(&bar_drain2);
      mbar_wait(&bar_drain2, 0, nullptr, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w serves TMEM lane quadrant w % 4 (rows 32 quad .. 32 quad + 31)
    // and key columns [64 part, 64 part + 64) of each 256-key tile; for the
    // O rescale and the epilogue it owns O columns [D/4 part, D/4 part + D/4).
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = a.scale_log2;
    if (part == 0) {
      // 1.0 for the ones rows of both V atoms, 2^-4 for P (the default mode
      // rewrites the P scale with each item's first P)
      tmem_st4(lane_base + C::kColOneA, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st4(lane_base + C::kColOneB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st4(lane_base + C::kColSfP, 0x7B7B7B7Bu, 0x7B7B7B7Bu, 0x7B7B7B7Bu, 0x7B7B7B7Bu);
      tmem_st_wait();
    }
    bool ok = true;
    uint32_t g = 0;  // ring iterations, counted across items
    int n_items = 0;
    FwdItem itm = item0;
    // next_item for a softmax warp: a warp-collective wait, lane 0 releases
    // the slot for the warp
    auto next_item_warp = [&](int n) -> bool {
      if constexpr (!PERSIST) {
        return false;
      } else {
        const bool got = warp_wait(&bar_clc[n & 1], (n >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax);
        uint32_t x = 0;
        const bool more = got && clc_query(&s_clc[n & 1], x);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_clc_free[n & 1]);
        if (!got) ok = false;
        return more && ok && fwd_item(a, x, itm);
      }
    };
    do {
    // every softmax warp has finished the previous item's epilogue: its O, L
    // columns and the s_l / s_mx buffers are free
    if (n_items >= 1 && !(ok = warp_wait(&bar_o_free, (n_items - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax)))
      break;
    int qt, hk, n_it, dh;
    int64_t nk, ktile_base;
    {
      const FwdGeo G = fwd_geo(a, itm);
      qt = itm.qt;
      hk = G.hk;
      n_it = G.n_it;
      dh = G.dh;
      nk = G.nk;
      ktile_base = itm.ktile_base;
    }
    const int64_t qpos = static_cast<int64_t>(qt) * 128 + r;  // document-relative query index
    float m = -INFINITY;  // running (lazy) max of the scaled scores, log2 units
    // O and L run on their own reference mo, at most kOLag binades behind m:
    // the P V MMA's A scale 2^(m - mo - 4) carries the difference, so a raise
    // of m rescales nothing in TMEM until the lag passes kOLag.  Scaling by a
    // power of two commutes with the fp32 sums, so O / L is the same.
    float mo = -INFINITY;
    float l16 = 0.0f;     // this warp's sum of 2^(s - m + 4) over its columns
    float ldiag = 0.0f;   // folded diagonal columns (FOLD): the weights their codes stand for
    for (int j = 0; j < n_it; ++j, ++g) {
      if (!(ok = warp_wait(&bar_s_full, g & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      // columns >= lim are masked (keys past the document end, or after the
      // query on the causal diagonal); only the last iteration has any
      int lim = 256;
      if (j == n_it - 1) {
        const int64_t rem = nk - static_cast<int64_t>(j) * 256;
        lim = rem < 256 ? static_cast<int>(rem) : 256;
        if (a.causal) {
          const int64_t c = qpos - static_cast<int64_t>(j) * 256 + 1;
          if (c < lim) lim = static_cast<int>(c);
        }
      }
      // a warp whose 64 columns are visible in all its rows takes their
      // maximum with the load itself
      const bool full = __all_sync(0xffffffffu, lim >= 64 * part + 64);
      float sv[64];
      float mt;
      if (full) {
        ld64_max(lane_base + C::kColS + 64 * part, sv, mt);
      } else {
        ld64(lane_base + C::kColS + 64 * part, sv);
      }
      // S is in registers: the next S MMA may start -- except on the folded
      // last iteration, whose diagonal half is read from TMEM again below
      // (the next S may be the next item's first)
      const bool hold_s = fold && j == n_it - 1;
      tc_fence_before();
      if (!hold_s) mbar_arrive(&bar_s_empty);
      if (!full) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = (64 * part + c < lim) ? sv[c] : -INFINITY;
        mt = max64(sv);
      }
      const int px = static_cast<int>(g & 1);
      s_mx[px][part][r] = mt;
      mbar_arrive(&bar_mx[px][quad]);
      if (!(ok = warp_wait(&bar_mx[px][quad], (g >> 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      mt = fmaxf(fmaxf(s_mx[px][0][r], s_mx[px][1][r]), fmaxf(s_mx[px][2][r], s_mx[px][3][r]));
      const float mts = mt * sl2;
      bool rescale_o = false, new_scale = j == 0;
      float factor = 1.0f, ofactor = 1.0f;
      // the reference stays on the integer grid of base-2 coordinates, so a
      // raise multiplies the earlier sums by an exact power of two and the
      // E4M3 weights are those of the final reference ceil(max) shifted by
      // whole binades (scale doubling, FLAMIA notes sec. 4)
      if (j == 0) {
        m = ceilf(mts);
        if constexpr (!FOLD) mo = m;
      } else if (mts > m + 4.0f) {
        const float mn = ceilf(mts);
        factor = exp2i_neg(static_cast<int>(fminf(mn - m, 127.0f)));
        m = mn;
        if constexpr (FOLD) {
          // the strict mode keeps O on m (its diagonal fold scales are
          // formed against m)
          ofactor = factor;
          rescale_o = true;
        } else {
          new_scale = true;
          if (m - mo > kOLag) {  // O and L catch up
            ofactor = exp2i_neg(static_cast<int>(fminf(m - mo, 127.0f)));
            mo = m;
            rescale_o = true;
          }
        }
      }
      const float neg = 4.0f - m;
      const uint64_t neg2 = f2_pack(neg, neg), sl2x2 = f2_pack(sl2, sl2);
      uint64_t lsa = 0, lsb = 0;  // four partial sums (+0.0) in two pairs
      uint32_t pw[16];  // E4M3 codes of this warp's 64 weights
      const bool diag = fold && j == n_it - 1 && (part >> 1) == dh;  // warp-uniform
      uint32_t sfb = 0u;
      if (!FOLD || !diag) {
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float2 x01 = f2_unpack(f2_fma(f2_pack(sv[c], sv[c + 1]), sl2x2, neg2));
          const float2 x23 = f2_unpack(f2_fma(f2_pack(sv[c + 2], sv[c + 3]), sl2x2, neg2));
          const float p0 = ex2_approx(x01.x), p1 = ex2_approx(x01.y);
          const float p2 = ex2_approx(x23.x), p3 = ex2_approx(x23.y);
          lsa = f2_add(lsa, f2_pack(p0, p1));
          lsb = f2_add(lsb, f2_pack(p2, p3));
          pw[c >> 2] = pack_e4m3x4(p0, p1, p2, p3);
        }
      } else if constexpr (FOLD) {
        // the 128 exponents of the diagonal tile (tile qt of this document),
        // 64 per column quarter; the sums run in units of 2^4 p like l16
        const uint8_t* kexp = a.vkey_sf + (static_cast<int64_t>(hk) * a.ntiles_k + ktile_base + qt) * 128 + 64 * (part & 1);
        const FoldOut fo = fold_keys(lane_base + C::kColS + 64 * part, 64 * part, lim, kexp, sl2x2, neg2, lsa, lsb);
#pragma unroll
        for (int k = 0; k < 16; ++k) pw[k] = fo.pw[k];
        sfb = fo.sfb;
        ldiag = fo.lw;
        lsa = fo.lsa;
        lsb = fo.lsb;
      }
      const float2 la = f2_unpack(lsa), lb = f2_unpack(lsb);
      const float lsum = (la.x + la.y) + (lb.x + lb.y);
      if (hold_s) {
        tc_fence_before();
        mbar_arrive(&bar_s_empty);
      }
      // the previous P V must be done before P is overwritten and O rescaled
      if (j > 0 && !(ok = warp_wait(&bar_o_done, (g - 1) & 1, abort_flag, a.err, kErrTimeoutSoftmax))) break;
      tc_fence_after();
      // tcgen05.ld/st are warp-collective: the whole warp rescales its rows'
      // share of O when any of them needs it (factor 1 for the others).
      if (__any_sync(0xffffffffu, rescale_o)) {
        const float factor = ofactor;
#pragma unroll
        for (int c = 0; c < D / 128; ++c) {
          const uint32_t col = C::kColO + (D / 4) * part + 32 * c;
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
        if (D == 64) {
          uint32_t rr[16];
          tmem_ld16(lane_base + C::kColO + 16 * part, rr);
          tmem_ld_wait();
          uint32_t w0[8], w1[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w0[k] = __float_as_uint(__uint_as_float(rr[k]) * factor);
            w1[k] = __float_as_uint(__uint_as_float(rr[8 + k]) * factor);
          }
          tmem_st8(lane_base + C::kColO + 16 * part, w0);
          tmem_st8(lane_base + C::kColO + 16 * part + 8, w1);
        }
        if (part == 0) {
          uint32_t rr[16];
          tmem_ld16(lane_base + C::kColL, rr);
          tmem_ld_wait();
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(rr[k]) * factor);
          tmem_st8(lane_base + C::kColL, w);
        }
      }
      {
        uint32_t w0[8], w1[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w0[k] = pw[k];
          w1[k] = pw[8 + k];
        }
        tmem_st8(lane_base + C::kColP + 16 * part, w0);
        tmem_st8(lane_base + C::kColP + 16 * part + 8, w1);
        // the P scale of row r sits at lane r, column base + r / 32, one byte
        // per K step: 2^(m - mo - 4) for all of them, rewritten when m or mo
        // moved (the previous P V, which read it, is done)
        if constexpr (!FOLD) {
          if (part == 0 && __any_sync(0xffffffffu, new_scale))
            tmem_st1(lane_base + C::kColSfP + quad, static_cast<uint32_t>(123.0f + (m - mo)) * 0x01010101u);
        }
        if (FOLD && diag) {
          // K steps 2 (part & 1) and 2 (part & 1) + 1 of the diagonal half: the
          // scale of row r at lane r, column base + r / 32, byte = sf_id (the
          // strict mode keeps O on m: no lag to carry)
          const uint32_t v = (part & 1) ? (0x00007F7Fu | (sfb << 16)) : (0x7F7F0000u | sfb);
          tmem_st1(lane_base + C::kColSfPd + 4 * (part & 1) + quad, v);
        }
      }
      l16 = l16 * factor + lsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_p_full);
    }
    // ---------------------------------------------------------- epilogue
    if (!ok) break;
    s_l[part][r] = l16;
    // the folded weights through the maxima buffer of the parity the last
    // iteration did not use (every warp of the quadrant read it before the
    // last iteration's max barrier)
    const int pu = static_cast<int>(g & 1);
    if (FOLD && fold) s_mx[pu][part][r] = ldiag;
    mbar_arrive(&bar_lsum);
    ok = role_wait(&bar_lsum, n_items & 1, abort_flag, a.err, kErrTimeoutEpilogue);
    if (ok) ok = role_wait(&bar_o_done, (g - 1) & 1, abort_flag, a.err, kErrTimeoutEpilogue);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    float inv;
    {
      uint32_t rr[16];
      tmem_ld16(lane_base + C::kColL, rr);
      tmem_ld_wait();
      float lq = __uint_as_float(rr[0]);
      if (FOLD && fold) lq += s_mx[pu][2 * dh][r] + s_mx[pu][2 * dh + 1][r];
      inv = 1.0f / lq;
    }
    const FwdGeo GE = fwd_geo(a, itm);  // the epilogue's own fields, recomputed
    const int h = itm.h;
    const bool valid = qpos < GE.n;
    const int64_t t = GE.doc_start + qpos;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (t * a.Hq + h) * D;
    constexpr int kCols = D / 4;  // 32 (d128) or 16 (d64) output channels per warp
    uint32_t rr[kCols];
    if constexpr (kCols == 32) {
      tmem_ld32(lane_base + C::kColO + kCols * part, rr);
    } else {
      tmem_ld16(lane_base + C::kColO + kCols * part, rr);
    }
    tmem_ld_wait();
    // O and L of this item are in registers: the next item's first P V may
    // restart them once every softmax warp is here
    tc_fence_before();
    mbar_arrive(&bar_o_free);
    if (valid) {
#pragma unroll
      for (int i = 0; i < kCols; i += 8) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(rr[i]) * inv, __uint_as_float(rr[i + 1]) * inv);
        v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * inv, __uint_as_float(rr[i + 3]) * inv);
        v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * inv, __uint_as_float(rr[i + 5]) * inv);
        v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * inv, __uint_as_float(rr[i + 7]) * inv);
        *reinterpret_cast<uint4*>(orow + kCols * part + i) = v;
      }
    }
    if (valid && part == 0)
      a.lse[static_cast<int64_t>(h) * a.T + t] =
          (m - 4.0f + log2f((s_l[0][r] + s_l[1][r]) + (s_l[2][r] + s_l[3][r]))) * 0.69314718055994531f;
    } while (next_item_warp(n_items++));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

namespace {

template <int D, bool FOLD, bool PERSIST>
cudaError_t launch_fwd_t(const FwdArgs& a, const FwdMaps& m, const dim3& grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, FOLD, PERSIST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<D, FOLD, PERSIST><<<grid, C::kThreads, C::kSmemBytes, stream>>>(m, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, const FwdMaps& m, const dim3& grid, bool fold, bool persist,
                         cudaStream_t stream) {
  if (persist) return fold ? launch_fwd_t<D, true, true>(a, m, grid, stream) : launch_fwd_t<D, false, true>(a, m, grid, stream);
  return fold ? launch_fwd_t<D, true, false>(a, m, grid, stream) : launch_fwd_t<D, false, false>(a, m, grid, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, int d, int max_seqlen, cudaStream_t stream) {
  // persistent (one CTA per SM runs at a time: the kernel holds all 512 TMEM
  // columns) over the virtual items -- with a cost-sorted list, or on equal
  // documents (heaviest query tiles first when causal); packed documents
  // without a list keep one CTA per slot of the max_seqlen grid, and so do
  // equal documents in strict mode (there the persistent variant measured
  // 9-14% slower)
  const bool fold = a.vkey_sf != nullptr && a.causal;
  const bool persist = a.items != nullptr || (a.cu_seqlens == nullptr && a.cu_k == nullptr && !fold);
  dim3 grid;
  if (persist) {  // one CTA per item; running CTAs take over the ones not yet started
    const int64_t total =
        a.items ? a.ntiles * a.Hq : static_cast<int64_t>(a.nq_tiles_doc) * a.num_docs * a.Hq;
    if (total <= 0 || total > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    grid = dim3(static_cast<unsigned>(total));
  } else {
    grid = dim3((max_seqlen + 127) / 128, a.num_docs, a.Hq);
  }
  return d == 128 ? launch_fwd_d<128>(a, m, grid, fold, persist, stream)
                  : launch_fwd_d<64>(a, m, grid, fold, persist, stream);
}

}  // namespace mxa
