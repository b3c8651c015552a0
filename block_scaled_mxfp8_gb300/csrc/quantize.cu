// quantize.cu -- bf16 -> MXFP8 quantizer (codes + UE8M0 scales), one pass.
//
// One CTA owns one (document, 128-token tile, head): it issues the loads of
// the tile's four 32-token groups (32 bytes per thread each) before any
// arithmetic, then quantizes the groups one after another, reading the bf16
// data once and writing every requested view:
//   ROW view  : one scale per 32 channels of a token (groups along d), the
//               view the Q K^T and dP = G V^T contractions use;
//   TOK view  : one scale per 32 document-relative tokens of a channel
//               (groups along tokens), the view P V, dV, dQ, dK use;
//   TOKBLOCK  : one scale for the whole 32 x d tile, written into both
//               layouts, one code set (FLAMIA notes sec. 3), optionally after
//               a normalized 128-point Hadamard rotation of each token.
// Scale rule: e = ceil(log2(amax / 448)) (FLAMIA notes sec. 4), computed
// exactly from the fp32 bits; codes are cvt.rn.satfinite E4M3 of x * 2^-e.
// Group max-abs, plain MX32 views (quantize_mx_kernel): in registers, one
// warp per 32-token group.  RMSNorm and token-block variants
// (quantize_kernel): within a token row by warp shuffles; along tokens by
// warp shuffles then one shared-memory pass across warps.
// Memory-bound: 2 B read + (1 + 1/32) B written per element per view.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa {

namespace {

constexpr uint32_t kInvSqrt128Bits = 0x3DB504F3u;  // fp32 nearest to 128^-1/2

template <int D>
struct QCfg {
  static constexpr int TPR = D / 16;            // threads per token row (16 channels each)
  static constexpr int kThreads = 32 * TPR;     // 32 rows
  static constexpr int kWarps = kThreads / 32;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One butterfly stage across threads: partner differs in chunk bit `bit`.
__device__ __forceinline__ void had_cross(float (&v)[16], int chunk, int lane_xor) {
  bool upper = ((chunk & lane_xor) == 0);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float other = __shfl_xor_sync(0xffffffffu, v[i], lane_xor);
    // upper element j: a + b with a = v[j] (mine), b = v[j+h] (partner)
    // lower element j+h: a - b with a = partner, b = mine
    v[i] = upper ? (v[i] + other) : (other - v[i]);
  }
}

}  // namespace

template <int D, bool TOKBLOCK, bool HAD>
__global__ void __launch_bounds__(QCfg<D>::kThreads) quantize_kernel(QuantArgs a) {
  using C = QCfg<D>;
  __shared__ float s_red[C::kWarps][D];
  __shared__ uint32_t s_red2[C::kWarps][D / 2];  // per-warp channel maxima, bf16 patterns, 2 per word
  __shared__ __align__(16) float s_sc[D];         // 2^-e of each channel
  __shared__ float s_blk[C::kWarps];
  __shared__ int64_t s_tile_base;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid / C::TPR;      // token row in a 32-token group
  const int chunk = tid % C::TPR;    // 16-channel chunk
  const int tile = blockIdx.x;       // 128-token tile inside the document
  const int b = blockIdx.y;          // document
  const int h = blockIdx.z;          // head

  int64_t doc_start, doc_len;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, doc_len);
  if (static_cast<int64_t>(tile) * 128 >= doc_len) return;  // past this document's last tile

  // the raw bf16 words of all four 32-token groups first: 4 x 32 bytes per
  // thread in flight before any arithmetic
  uint4 raw[4][2];
#pragma unroll
  for (int gq = 0; gq < 4; ++gq) {
    const int64_t tok = static_cast<int64_t>(tile) * 128 + gq * 32 + row;
    if (tok < doc_len) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) +
                                                        ((doc_start + tok) * a.H + h) * D + chunk * 16);
      raw[gq][0] = __ldg(src);
      raw[gq][1] = __ldg(src + 1);
    } else {
      raw[gq][0] = make_uint4(0u, 0u, 0u, 0u);
      raw[gq][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // First scale tile of this document (each document owns ceil(n / 128)
  // consecutive 128-token tiles in the [H, NT, 512] scale layouts).
  if (a.cu_seqlens == nullptr) {
    if (tid == 0) s_tile_base = static_cast<int64_t>(b) * ((doc_len + 127) / 128);
  } else {
    int64_t part = 0;
    for (int i = tid; i < b; i += C::kThreads) part += (a.cu_seqlens[i + 1] - a.cu_seqlens[i] + 127) / 128;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (tid == 0) s_tile_base = 0;
    __syncthreads();
    if (lane == 0 && part) atomicAdd(reinterpret_cast<unsigned long long*>(&s_tile_base), static_cast<unsigned long long>(part));
  }
  __syncthreads();
  const int64_t atom_base = (static_cast<int64_t>(h) * a.ntiles + s_tile_base + tile) * kAtomBytes;

#pragma unroll
  for (int gq = 0; gq < 4; ++gq) {
    const int g = tile * 4 + gq;  // 32-token group inside the document
    const int64_t t = doc_start + static_cast<int64_t>(g) * 32 + row;
    const bool valid = (static_cast<int64_t>(g) * 32 + row) < doc_len;
    const int64_t elem0 = (t * a.H + h) * D + chunk * 16;

    float v[16];
    {
      const uint32_t w[8] = {raw[gq][0].x, raw[gq][0].y, raw[gq][0].z, raw[gq][0].w,
                             raw[gq][1].x, raw[gq][1].y, raw[gq][1].z, raw[gq][1].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
      }
    }

    if (a.rms) {
      // RMSNorm in IEEE fp32, in a fixed order: this thread's 16 squares in
      // channel order, then the TPR partial sums of the row pairwise (xor 1, 2,
      // 4: every lane of the row ends with the same tree sum); r = 1 / sqrt(s /
      // d + eps) with correctly rounded sqrt and division (0 when s / d + eps
      // is 0); y = (x * r) * w.  (FA4 write-up, "Fused RMSNorm+Quantize".)
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ss = __fadd_rn(ss, __fmul_rn(v[i], v[i]));
#pragma unroll
      for (int o = 1; o < C::TPR; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      const float den = __fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), a.rms_eps);
      const float r = den == 0.0f ? 0.0f : __fdiv_rn(1.0f, __fsqrt_rn(den));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float t = __fmul_rn(v[i], r);
        v[i] = a.rms_w ? __fmul_rn(t, __ldg(a.rms_w + chunk * 16 + i)) : t;
      }
    }

    if constexpr (HAD) {
      // Sylvester order: in-thread stages h = 1, 2, 4, 8, then across the 8
      // threads of the row for h = 16, 32, 64 (chunk bits 0, 1, 2).
#pragma unroll
      for (int hh = 1; hh < 16; hh *= 2) {
#pragma unroll
        for (int i = 0; i < 16; i += 2 * hh) {
#pragma unroll
          for (int j = i; j < i + hh; ++j) {
            float x0 = v[j], x1 = v[j + hh];
            v[j] = x0 + x1;
            v[j + hh] = x0 - x1;
          }
        }
      }
      had_cross(v, chunk, 1);
      had_cross(v, chunk, 2);
      had_cross(v, chunk, 4);
      const float r = __uint_as_float(kInvSqrt128Bits);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], r);
    }

    // max-abs of this thread's 16 values in independent chains
    float amax_local = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                             fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
    amax_local = fmaxf(amax_local, fmaxf(fmaxf(fmaxf(fabsf(v[8]), fabsf(v[9])), fmaxf(fabsf(v[10]), fabsf(v[11]))),
                                         fmaxf(fmaxf(fabsf(v[12]), fabsf(v[13])), fmaxf(fabsf(v[14]), fabsf(v[15])))));

    if constexpr (TOKBLOCK) {
      // one exponent for the whole tile
      float m = amax_local;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) s_blk[warp] = m;
      __syncthreads();
      float bm = 0.0f;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) bm = fmaxf(bm, s_blk[w]);
      const int e = mx_exponent_bits(__float_as_uint(bm));
      const float sc = exp2i_neg(e);
      const uint8_t eb = static_cast<uint8_t>(e + 127);
      if (valid) {
        uint4 out;
        out.x = pack_e4m3x4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
        out.y = pack_e4m3x4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
        out.z = pack_e4m3x4(v[8] * sc, v[9] * sc, v[10] * sc, v[11] * sc);
        out.w = pack_e4m3x4(v[12] * sc, v[13] * sc, v[14] * sc, v[15] * sc);
        *reinterpret_cast<uint4*>(a.row_codes + elem0) = out;
        if ((chunk & 1) == 0) a.row_scales[atom_base + row * 16 + (g & 3) * 4 + chunk / 2] = eb;
      }
      if (tid < D) a.tok_scales[atom_base + atom_offset(tid, g & 3)] = eb;
      __syncthreads();  // s_blk is rewritten by the next group
      continue;
    } else {
      if (a.write_row) {
        float m = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, 1));  // 32-channel group
        const int e = mx_exponent_bits(__float_as_uint(m));
        const float sc = exp2i_neg(e);
        if (valid) {
          uint4 out;
          out.x = pack_e4m3x4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
          out.y = pack_e4m3x4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
          out.z = pack_e4m3x4(v[8] * sc, v[9] * sc, v[10] * sc, v[11] * sc);
          out.w = pack_e4m3x4(v[12] * sc, v[13] * sc, v[14] * sc, v[15] * sc);
          *reinterpret_cast<uint4*>(a.row_codes + elem0) = out;
          if ((chunk & 1) == 0) a.row_scales[atom_base + row * 16 + (g & 3) * 4 + chunk / 2] = static_cast<uint8_t>(e + 127);
        }
      }
      if (a.write_tok) {
        // per-channel max over the 32 rows: rows of a warp differ in the lane
        // bits above log2(TPR); then across warps in shared memory.
        if (!a.rms) {
          // on the bf16 bit patterns: |x| is the pattern without its sign
          // bit, and the patterns of non-negative values order as unsigned
          // integers, so one halfword max serves two channels
          uint32_t m2[8] = {raw[gq][0].x & 0x7FFF7FFFu, raw[gq][0].y & 0x7FFF7FFFu, raw[gq][0].z & 0x7FFF7FFFu,
                            raw[gq][0].w & 0x7FFF7FFFu, raw[gq][1].x & 0x7FFF7FFFu, raw[gq][1].y & 0x7FFF7FFFu,
                            raw[gq][1].z & 0x7FFF7FFFu, raw[gq][1].w & 0x7FFF7FFFu};
#pragma unroll
          for (int o = C::TPR; o < 32; o <<= 1) {
#pragma unroll
            for (int k = 0; k < 8; ++k) m2[k] = __vmaxu2(m2[k], __shfl_xor_sync(0xffffffffu, m2[k], o));
          }
          if (lane < C::TPR) {
#pragma unroll
            for (int k = 0; k < 8; ++k) s_red2[warp][chunk * 8 + k] = m2[k];
          }
          __syncthreads();
          if (tid < D / 2) {  // channels 2 tid (low halfword) and 2 tid + 1 (high)
            uint32_t mm = 0u;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) mm = __vmaxu2(mm, s_red2[w][tid]);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int ch = 2 * tid + hf;
              const int e = mx_exponent_bits(hf ? (mm & 0xFFFF0000u) : (mm << 16));
              s_sc[ch] = exp2i_neg(e);
              a.tok_scales[atom_base + atom_offset(ch, g & 3)] = static_cast<uint8_t>(e + 127);
            }
          }
        } else {
          float cm[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float m = fabsf(v[i]);
#pragma unroll
            for (int o = C::TPR; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            cm[i] = m;
          }
          if (lane < C::TPR) {
#pragma unroll
            for (int i = 0; i < 16; ++i) s_red[warp][chunk * 16 + i] = cm[i];
          }
          __syncthreads();
          if (tid < D) {
            float m = 0.0f;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) m = fmaxf(m, s_red[w][tid]);
            const int e = mx_exponent_bits(__float_as_uint(m));
            s_sc[tid] = exp2i_neg(e);
            a.tok_scales[atom_base + atom_offset(tid, g & 3)] = static_cast<uint8_t>(e + 127);
          }
        }
        __syncthreads();
        if (valid) {
          float y[16];
          const float4* sc4 = reinterpret_cast<const float4*>(s_sc + chunk * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 f = sc4[i];
            y[4 * i] = v[4 * i] * f.x;
            y[4 * i + 1] = v[4 * i + 1] * f.y;
            y[4 * i + 2] = v[4 * i + 2] * f.z;
            y[4 * i + 3] = v[4 * i + 3] * f.w;
          }
          uint4 out;
          out.x = pack_e4m3x4(y[0], y[1], y[2], y[3]);
          out.y = pack_e4m3x4(y[4], y[5], y[6], y[7]);
          out.z = pack_e4m3x4(y[8], y[9], y[10], y[11]);
          out.w = pack_e4m3x4(y[12], y[13], y[14], y[15]);
          *reinterpret_cast<uint4*>(a.tok_codes + elem0) = out;
        }
        __syncthreads();  // s_red / s_sc are rewritten by the next group
      }
    }
  }  // 32-token groups
}

// ------------------------------------------------------- MX32, ROW/TOK views
// The plain MX32 path (no RMSNorm, no token blocks), laid out so that both
// group maxima stay in registers: one CTA per (head, 128-token tile,
// document), one warp per 32-token group.  Lane l holds channels
// [16 c, 16 c + 16), c = l % LPR, of the group's tokens l / LPR + k RPI
// (k < TPL): two warp-wide 16-byte loads cover RPI whole token rows, so loads
// and the 16-byte code stores stay coalesced.  Pass 1, the maxima: TOK view,
// per channel over the group, a register loop over the lane's TPL tokens on
// the bf16 bit patterns (two channels per halfword max) plus shuffles across
// the lanes of the same channels; ROW view, per token over 32 channels, the
// lane's 16 channels plus one shuffle (the 2 lanes of the 32-channel group),
// two tokens per shuffled word.  Pass 2, one token at a time: its 16 values
// are unpacked once and scaled (packed fp32x2 multiplies by powers of two)
// into both views.  No shared memory, no block barrier after the tile base;
// all loads are issued before any arithmetic.  Every byte of the CTA's scale
// atoms is written, padding included (0x7F: rows past the document end, the
// groups and rows beyond d = 64).
template <int D>
__global__ void __launch_bounds__(128, 5) quantize_mx_kernel(QuantArgs a) {
  constexpr int LPR = D / 16;    // lanes per token row
  constexpr int RPI = 32 / LPR;  // token rows per warp load
  constexpr int TPL = 32 / RPI;  // tokens per lane
  __shared__ int64_t s_tile_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cl = lane % LPR, rl = lane / LPR;
  // head fastest: CTAs that run together read and write whole token rows
  // (all heads of a token are contiguous) instead of 8 KB-strided pieces
  const int h = blockIdx.x, tile = blockIdx.y, b = blockIdx.z;
  int64_t doc_start, doc_len;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, doc_len);
  if (static_cast<int64_t>(tile) * 128 >= doc_len) return;
  const int64_t tok0 = static_cast<int64_t>(tile) * 128 + warp * 32;  // the group's first token (document-relative)

  uint4 raw[TPL][2];
#pragma unroll
  for (int k = 0; k < TPL; ++k) {
    const int64_t pos = tok0 + rl + k * RPI;
    if (pos < doc_len) {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) +
                                                        ((doc_start + pos) * a.H + h) * D + cl * 16);
      raw[k][0] = __ldg(src);
      raw[k][1] = __ldg(src + 1);
    } else {
      raw[k][0] = raw[k][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // first scale tile of this document
  if (a.cu_seqlens == nullptr) {
    if (tid == 0) s_tile_base = static_cast<int64_t>(b) * ((doc_len + 127) / 128);
  } else {
    int64_t part = 0;
    for (int i = tid; i < b; i += 128) part += (a.cu_seqlens[i + 1] - a.cu_seqlens[i] + 127) / 128;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (tid == 0) s_tile_base = 0;
    __syncthreads();
    if (lane == 0 && part) atomicAdd(reinterpret_cast<unsigned long long*>(&s_tile_base), static_cast<unsigned long long>(part));
  }
  __syncthreads();
  const int64_t atom_base = (static_cast<int64_t>(h) * a.ntiles + s_tile_base + tile) * kAtomBytes;

  // ---- pass 1: TOK view channel maxima -> this lane's 16 channel scales
  uint64_t sct[8];  // (2^-e of channel 2 i, 2^-e of channel 2 i + 1) as fp32x2
  if (a.write_tok) {
    uint32_t m[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // |x| patterns, channels (2 i, 2 i + 1) of the lane
#pragma unroll
    for (int k = 0; k < TPL; ++k) {
      m[0] = __vmaxu2(m[0], raw[k][0].x & 0x7FFF7FFFu);
      m[1] = __vmaxu2(m[1], raw[k][0].y & 0x7FFF7FFFu);
      m[2] = __vmaxu2(m[2], raw[k][0].z & 0x7FFF7FFFu);
      m[3] = __vmaxu2(m[3], raw[k][0].w & 0x7FFF7FFFu);
      m[4] = __vmaxu2(m[4], raw[k][1].x & 0x7FFF7FFFu);
      m[5] = __vmaxu2(m[5], raw[k][1].y & 0x7FFF7FFFu);
      m[6] = __vmaxu2(m[6], raw[k][1].z & 0x7FFF7FFFu);
      m[7] = __vmaxu2(m[7], raw[k][1].w & 0x7FFF7FFFu);
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) m[i] = __vmaxu2(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e0 = mx_exponent_bits(m[i] << 16), e1 = mx_exponent_bits(m[i] & 0xFFFF0000u);
      sct[i] = f2_pack(exp2i_neg(e0), exp2i_neg(e1));
      if (rl == 0) {
        a.tok_scales[atom_base + atom_offset(cl * 16 + 2 * i, warp)] = static_cast<uint8_t>(e0 + 127);
        a.tok_scales[atom_base + atom_offset(cl * 16 + 2 * i + 1, warp)] = static_cast<uint8_t>(e1 + 127);
        if (D < 128) {  // atom rows D .. 127 are padding
          a.tok_scales[atom_base + atom_offset(D + cl * 16 + 2 * i, warp)] = 0x7F;
          a.tok_scales[atom_base + atom_offset(D + cl * 16 + 2 * i + 1, warp)] = 0x7F;
        }
      }
    }
  }
  // ---- pass 1: ROW view token maxima, two tokens per word
  uint32_t pk[TPL / 2];
  if (a.write_row) {
#pragma unroll
    for (int k = 0; k < TPL; k += 2) {
      uint32_t t2[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint4 r0 = raw[k + j][0], r1 = raw[k + j][1];
        const uint32_t w = __vmaxu2(__vmaxu2(__vmaxu2(r0.x & 0x7FFF7FFFu, r0.y & 0x7FFF7FFFu),
                                             __vmaxu2(r0.z & 0x7FFF7FFFu, r0.w & 0x7FFF7FFFu)),
                                    __vmaxu2(__vmaxu2(r1.x & 0x7FFF7FFFu, r1.y & 0x7FFF7FFFu),
                                             __vmaxu2(r1.z & 0x7FFF7FFFu, r1.w & 0x7FFF7FFFu)));
        t2[j] = max(w & 0xFFFFu, w >> 16);
      }
      pk[k / 2] = t2[0] | (t2[1] << 16);
    }
#pragma unroll
    for (int k = 0; k < TPL / 2; ++k) pk[k] = __vmaxu2(pk[k], __shfl_xor_sync(0xffffffffu, pk[k], 1));
  }

  // ---- pass 2: each token's 16 values once, into both views
#pragma unroll
  for (int k = 0; k < TPL; ++k) {
    const int lt = rl + k * RPI;  // token inside the group
    const int64_t pos = tok0 + lt;
    const bool valid = pos < doc_len;
    const int64_t off = ((doc_start + pos) * a.H + h) * D + cl * 16;
    const uint32_t wv[8] = {raw[k][0].x, raw[k][0].y, raw[k][0].z, raw[k][0].w,
                            raw[k][1].x, raw[k][1].y, raw[k][1].z, raw[k][1].w};
    uint64_t x2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x2[i] = f2_pack(bf16_lo(wv[i]), bf16_hi(wv[i]));
    if (a.write_tok && valid) {
      uint32_t q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 y0 = f2_unpack(f2_mul(x2[2 * i], sct[2 * i]));
        const float2 y1 = f2_unpack(f2_mul(x2[2 * i + 1], sct[2 * i + 1]));
        q[i] = pack_e4m3x4(y0.x, y0.y, y1.x, y1.y);
      }
      *reinterpret_cast<uint4*>(a.tok_codes + off) = make_uint4(q[0], q[1], q[2], q[3]);
    }
    if (a.write_row) {
      const uint32_t mb = (k & 1) ? (pk[k / 2] & 0xFFFF0000u) : (pk[k / 2] << 16);
      const int e = mx_exponent_bits(mb);
      const float sc = exp2i_neg(e);
      if (valid) {
        const uint64_t sc2 = f2_pack(sc, sc);
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 y0 = f2_unpack(f2_mul(x2[2 * i], sc2));
          const float2 y1 = f2_unpack(f2_mul(x2[2 * i + 1], sc2));
          q[i] = pack_e4m3x4(y0.x, y0.y, y1.x, y1.y);
        }
        *reinterpret_cast<uint4*>(a.row_codes + off) = make_uint4(q[0], q[1], q[2], q[3]);
      }
      if ((cl & 1) == 0) {
        uint8_t* rs = a.row_scales + atom_base + lt * 16 + warp * 4;
        rs[cl / 2] = valid ? static_cast<uint8_t>(e + 127) : 0x7F;
        if (D < 128) rs[cl / 2 + D / 32] = 0x7F;  // groups D / 32 .. 3 are padding
      }
    }
  }
}

// ------------------------------------------------------------ per-key view
// FLAMIA notes sec. 4 (moving the scale across the boundary): on the causal
// diagonal tile each key's V row gets its own power-of-two scale, which the
// forward folds into the probability operand.  The view: e_t by the MX rule
// over all d channels of token t and head h, codes E4M3(x * 2^-e_t).  One CTA
// per (128-token tile, document, head); D / 8 threads per token row, 8
// channels each.
template <int D>
__global__ void __launch_bounds__(256) quantize_key_kernel(KeyQuantArgs a) {
  constexpr int TPR = D / 8;
  constexpr int RPP = 256 / TPR;  // rows per pass
  __shared__ int64_t s_slot;
  const int tid = threadIdx.x, row0 = tid / TPR, chunk = tid % TPR;
  const int tile = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
  int64_t doc_start, n;
  doc_bounds(a.cu_seqlens, a.num_docs, a.T, b, doc_start, n);
  if (static_cast<int64_t>(tile) * 128 >= n) return;
  // first scale tile of this document (a sum of ceil(n / 128) over the
  // earlier documents)
  if (a.cu_seqlens == nullptr) {
    if (tid == 0) s_slot = static_cast<int64_t>(b) * ((n + 127) / 128);
  } else {
    int64_t part = 0;
    for (int i = tid; i < b; i += 256) part += (a.cu_seqlens[i + 1] - a.cu_seqlens[i] + 127) / 128;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (tid == 0) s_slot = 0;
    __syncthreads();
    if ((tid & 31) == 0 && part) atomicAdd(reinterpret_cast<unsigned long long*>(&s_slot), static_cast<unsigned long long>(part));
  }
  __syncthreads();
  const int64_t tb = s_slot;
  uint4 raw[128 / RPP];
#pragma unroll
  for (int i = 0; i < 128 / RPP; ++i) {
    const int64_t pos = static_cast<int64_t>(tile) * 128 + row0 + i * RPP;
    raw[i] = pos < n ? __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) +
                                                            ((doc_start + pos) * a.H + h) * D + chunk * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 128 / RPP; ++i) {
    const int r = row0 + i * RPP;
    const int64_t pos = static_cast<int64_t>(tile) * 128 + r;
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float v[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = bf16_lo(w[k]);
      v[2 * k + 1] = bf16_hi(w[k]);
    }
    float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                    fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
    for (int o = TPR / 2; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));  // the row's lanes
    const int e = mx_exponent_bits(__float_as_uint(m));
    const float sc = exp2i_neg(e);
    if (pos < n) {
      uint2 out;
      out.x = pack_e4m3x4(v[0] * sc, v[1] * sc, v[2] * sc, v[3] * sc);
      out.y = pack_e4m3x4(v[4] * sc, v[5] * sc, v[6] * sc, v[7] * sc);
      *reinterpret_cast<uint2*>(a.codes + ((doc_start + pos) * a.H + h) * D + chunk * 8) = out;
      if (chunk == 0) a.scales[(static_cast<int64_t>(h) * a.ntiles + tb + tile) * 128 + r] = static_cast<uint8_t>(e + 127);
    }
  }
}

cudaError_t launch_quantize_key(const KeyQuantArgs& a, int d, int max_seqlen, cudaStream_t stream) {
  const dim3 grid((max_seqlen + 127) / 128, a.num_docs, a.H);
  if (d == 128) quantize_key_kernel<128><<<grid, 256, 0, stream>>>(a);
  else quantize_key_kernel<64><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantArgs& a, int d, bool tokblock, bool hadamard, int max_groups,
                            cudaStream_t stream) {
  dim3 grid((max_groups + 3) / 4, a.num_docs, a.H);  // one CTA per 128-token tile
  if (!tokblock && !a.rms) {  // the plain MX32 views: register-resident group maxima
    const dim3 g2(a.H, (max_groups + 3) / 4, a.num_docs);
    if (d == 128) quantize_mx_kernel<128><<<g2, 128, 0, stream>>>(a);
    else quantize_mx_kernel<64><<<g2, 128, 0, stream>>>(a);
    return cudaGetLastError();
  }
  if (d == 128) {
    constexpr int nt = QCfg<128>::kThreads;
    if (tokblock && hadamard)
      quantize_kernel<128, true, true><<<grid, nt, 0, stream>>>(a);
    else if (tokblock)
      quantize_kernel<128, true, false><<<grid, nt, 0, stream>>>(a);
    else
      quantize_kernel<128, false, false><<<grid, nt, 0, stream>>>(a);
  } else {
    constexpr int nt = QCfg<64>::kThreads;
    if (tokblock)
      quantize_kernel<64, true, false><<<grid, nt, 0, stream>>>(a);
    else
      quantize_kernel<64, false, false><<<grid, nt, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mxa
