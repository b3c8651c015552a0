// api.cu -- the C ABI of libmxa.so (declared in include/mxa.h): argument
// validation, TMA tensor-map encoding and kernel launches.  Nothing here
// allocates device memory; every buffer belongs to the caller.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mxa.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace mxa {

// Device error word written by kernels whose bounded waits ran out.
static __device__ int g_err_word;

static int* g_err_ptr[64];
static std::mutex g_mu;

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over E4M3 codes [T, H, d]: box of 128 tokens x 1 head x d bytes,
// swizzled to the tensor core's K-major / MN-major layout.
bool make_code_map(CUtensorMap* map, const void* codes, int64_t T, int H, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(codes), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool is_cross(const mxa_shape& s) { return s.T_k != 0; }

// Most 128-token tiles in one document (query side).
int64_t max_doc_tiles(const mxa_shape& s) {
  const int64_t maxlen = s.cu_seqlens ? s.max_seqlen : (s.num_docs > 0 ? s.T / s.num_docs : 0);
  return (maxlen + 127) / 128;
}

// The two sides of a call: queries, and keys/values (the same for
// self-attention).
Side q_side(const mxa_shape& s) {
  return Side{s.cu_seqlens, s.T, s.ntiles, static_cast<int>(max_doc_tiles(s))};
}
Side k_side(const mxa_shape& s) {
  if (!is_cross(s)) return q_side(s);
  const int64_t maxlen = s.cu_seqlens_k ? s.max_seqlen_k : (s.num_docs > 0 ? s.T_k / s.num_docs : 0);
  return Side{s.cu_seqlens_k, s.T_k, s.ntiles_k, static_cast<int>((maxlen + 127) / 128)};
}

// Longest document of either side, in tokens (sizes the grids).
int max_len(const mxa_shape& s) {
  const Side q = q_side(s), k = k_side(s);
  return static_cast<int>(128 * (q.max_tiles > k.max_tiles ? q.max_tiles : k.max_tiles));
}

// Bytes of the tile-padded D and LSE rows (both backward paths).
size_t bwd_rows_bytes(const mxa_shape& s) {
  return 2 * static_cast<size_t>(s.Hq) * static_cast<size_t>(s.ntiles > 0 ? s.ntiles : 0) * 128 * 4;
}

// Bytes of the emitted dS (16 KB of codes + 16 block scales per tile pair,
// or a 512-byte scale atom per pair for the strict dQ operand).
size_t bwd_ds_bytes(const mxa_shape& s, bool strict = false) {
  const int64_t ntk = k_side(s).ntiles;
  return static_cast<size_t>(s.Hq) * static_cast<size_t>(ntk > 0 ? ntk : 0) *
         static_cast<size_t>(max_doc_tiles(s)) * (16384 + (strict ? kAtomBytes : 16));
}

// Bytes of one side's cost-sorted tile list.
size_t list_bytes(const mxa_shape& s, const Side& sd) {
  return tile_list_bytes(s.num_docs, sd.ntiles > 0 ? sd.ntiles : 0);
}

// Whether the attention kernels take their CTAs from the tile lists: packed
// documents or cross-attention (equal self-attention documents fill the
// max_seqlen grid exactly, in the same order), no document longer than the
// list builder's limit, and grids of NT x heads CTAs that fit one dimension.
bool uses_list(const mxa_shape& s) {
  const Side q = q_side(s), k = k_side(s);
  return (s.cu_seqlens != nullptr || is_cross(s)) && tile_lists_supported(q.max_tiles) &&
         tile_lists_supported(k.max_tiles) && q.ntiles * static_cast<int64_t>(s.Hq) <= 0x7FFFFFFFll &&
         k.ntiles * static_cast<int64_t>(s.Hkv) <= 0x7FFFFFFFll;
}

mxa_status check_view(const mxa_qview& v) {
  if (!v.codes || !v.scales) return MXA_ERR_ARG;
  if (!aligned(v.codes, 16) || !aligned(v.scales, 16)) return MXA_ERR_ALIGN;
  return MXA_OK;
}

mxa_status check_shape(const mxa_shape& s) {
  if (s.T < 0 || s.T > 0x7FFFFFFFll) return MXA_ERR_ARG;
  if (s.Hq <= 0 || s.Hkv <= 0 || s.num_docs <= 0 || s.ntiles <= 0 || s.max_seqlen <= 0) return MXA_ERR_ARG;
  if (s.num_docs > 65535 || s.Hq > 65535) return MXA_ERR_ARG;
  if (s.d != 64 && s.d != 128) return MXA_ERR_UNSUPPORTED;
  if (s.Hq % s.Hkv != 0) return MXA_ERR_UNSUPPORTED;
  if (!s.cu_seqlens && (s.T % s.num_docs != 0 || s.T / s.num_docs > s.max_seqlen)) return MXA_ERR_ARG;
  if (!(s.softmax_scale >= 0.0f) || !std::isfinite(s.softmax_scale)) return MXA_ERR_ARG;
  if (is_cross(s)) {
    if (s.T_k < 0 || s.T_k > 0x7FFFFFFFll || s.ntiles_k <= 0 || s.max_seqlen_k <= 0) return MXA_ERR_ARG;
    if (!s.cu_seqlens_k && (s.T_k % s.num_docs != 0 || s.T_k / s.num_docs > s.max_seqlen_k)) return MXA_ERR_ARG;
    if (s.causal) return MXA_ERR_UNSUPPORTED;
  }
  return MXA_OK;
}

// Key/value side of the kernel arguments.
template <class A>
void set_k_side(A& a, const mxa_shape& s) {
  const Side k = k_side(s);
  a.Tk = k.T;
  a.cu_k = k.cu;
  a.ntiles_k = k.ntiles;
}

float alpha_of(const mxa_shape& s) { return s.softmax_scale > 0.0f ? s.softmax_scale : 1.0f / std::sqrt(static_cast<float>(s.d)); }

}  // namespace
}  // namespace mxa

using namespace mxa;

extern "C" {

int mxa_abi_version(void) { return MXA_ABI_VERSION; }

const char* mxa_status_str(mxa_status s) {
  switch (s) {
    case MXA_OK: return "ok";
    case MXA_ERR_ARG: return "invalid argument";
    case MXA_ERR_ALIGN: return "misaligned buffer";
    case MXA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MXA_ERR_WORKSPACE: return "workspace too small";
    case MXA_ERR_CUDA: return "CUDA error";
    case MXA_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

int64_t mxa_scale_tiles(int64_t T, int num_docs, const int32_t* cu) {
  if (T < 0 || num_docs <= 0) return -1;
  if (!cu) {
    if (T % num_docs) return -1;
    return static_cast<int64_t>(num_docs) * ((T / num_docs + 127) / 128);
  }
  int64_t nt = 0;
  if (cu[0] != 0 || cu[num_docs] != T) return -1;
  for (int b = 0; b < num_docs; ++b) {
    const int64_t n = static_cast<int64_t>(cu[b + 1]) - cu[b];
    if (n < 0) return -1;
    nt += (n + 127) / 128;
  }
  return nt;
}

int64_t mxa_scale_tiles_bound(int64_t T, int num_docs) {
  if (T < 0 || num_docs <= 0) return -1;
  return (T + 127) / 128 + num_docs;
}

size_t mxa_scale_bytes(int H, int64_t ntiles) {
  if (H <= 0 || ntiles < 0) return 0;
  return static_cast<size_t>(H) * static_cast<size_t>(ntiles) * kAtomBytes;
}

size_t mxa_key_scale_bytes(int H, int64_t ntiles) {
  if (H <= 0 || ntiles < 0) return 0;
  return static_cast<size_t>(H) * static_cast<size_t>(ntiles) * 128;
}

}  // extern "C"

namespace {

mxa_status quantize_impl(const void* x, int64_t T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                         int max_seqlen, int64_t ntiles, mxa_scale_mode mode, int views, int hadamard,
                         mxa_qview* row, mxa_qview* tok, int rms, const float* rms_w, float rms_eps,
                         cudaStream_t stream) {
  if (!x || T < 0 || T > 0x7FFFFFFFll || H <= 0 || H > 65535 || num_docs <= 0 || num_docs > 65535 ||
      ntiles <= 0 || max_seqlen <= 0)
    return MXA_ERR_ARG;
  if (d != 64 && d != 128) return MXA_ERR_UNSUPPORTED;
  if (!cu_seqlens && (T % num_docs != 0 || T / num_docs > max_seqlen)) return MXA_ERR_ARG;
  if (!aligned(x, 16)) return MXA_ERR_ALIGN;
  const bool tokblock = mode == MXA_SCALE_TOKBLOCK32;
  if (mode != MXA_SCALE_MX32 && !tokblock) return MXA_ERR_ARG;
  if (views <= 0 || (views & ~(MXA_VIEW_ROW | MXA_VIEW_TOK))) return MXA_ERR_ARG;
  if (hadamard && (!tokblock || d != 128)) return MXA_ERR_UNSUPPORTED;
  const bool w_row = (views & MXA_VIEW_ROW) != 0, w_tok = (views & MXA_VIEW_TOK) != 0;
  if (tokblock) {
    if (!(w_row && w_tok) || !row || !tok || !row->codes || !row->scales || !tok->scales) return MXA_ERR_ARG;
    if (tok->codes && tok->codes != row->codes) return MXA_ERR_ARG;
    if (!aligned(row->codes, 16) || !aligned(row->scales, 16) || !aligned(tok->scales, 16)) return MXA_ERR_ALIGN;
  } else {
    if (w_row) {
      if (!row) return MXA_ERR_ARG;
      mxa_status st = check_view(*row);
      if (st != MXA_OK) return st;
    }
    if (w_tok) {
      if (!tok) return MXA_ERR_ARG;
      mxa_status st = check_view(*tok);
      if (st != MXA_OK) return st;
    }
  }
  if (T == 0) return MXA_OK;
  // The plain MX32 kernel writes every byte of the scale atoms it owns
  // (padding included); atoms no CTA owns exist only when ntiles exceeds the
  // documents' tiles (an upper bound), which the host can rule out for equal
  // documents only.  Every other call fills the layouts with 0x7F first.
  const bool plain = !tokblock && !rms;
  const bool exact_nt = !cu_seqlens && ntiles == static_cast<int64_t>(num_docs) * ((T / num_docs + 127) / 128);
  if (!(plain && exact_nt)) {
    const size_t sbytes = mxa_scale_bytes(H, ntiles);
    if ((w_row || tokblock) && cudaMemsetAsync(row->scales, 0x7F, sbytes, stream) != cudaSuccess)
      return MXA_ERR_CUDA;
    if ((w_tok || tokblock) && cudaMemsetAsync(tok->scales, 0x7F, sbytes, stream) != cudaSuccess)
      return MXA_ERR_CUDA;
  }
  QuantArgs a{};
  a.x = x;
  a.T = T;
  a.H = H;
  a.cu_seqlens = cu_seqlens;
  a.num_docs = num_docs;
  a.ntiles = ntiles;
  a.write_row = w_row || tokblock;
  a.write_tok = w_tok || tokblock;
  a.row_codes = (w_row || tokblock) ? row->codes : nullptr;
  a.row_scales = (w_row || tokblock) ? row->scales : nullptr;
  a.tok_codes = (w_tok && !tokblock) ? tok->codes : nullptr;
  a.tok_scales = (w_tok || tokblock) ? tok->scales : nullptr;
  a.rms = rms;
  a.rms_w = rms_w;
  a.rms_eps = rms_eps;
  const int max_groups = (cu_seqlens ? max_seqlen : static_cast<int>(T / num_docs)) + 31;
  if (launch_quantize(a, d, tokblock, hadamard != 0, max_groups / 32, stream) != cudaSuccess) return MXA_ERR_CUDA;
  return MXA_OK;
}

}  // namespace

extern "C" {

mxa_status mxa_quantize(const void* x, int64_t T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                        int max_seqlen, int64_t ntiles, mxa_scale_mode mode, int views, int hadamard,
                        mxa_qview* row, mxa_qview* tok, cudaStream_t stream) {
  return quantize_impl(x, T, H, d, cu_seqlens, num_docs, max_seqlen, ntiles, mode, views, hadamard, row, tok, 0,
                       nullptr, 0.0f, stream);
}

mxa_status mxa_rmsnorm_quantize(const void* x, const float* weight, float eps, int64_t T, int H, int d,
                                const int32_t* cu_seqlens, int num_docs, int max_seqlen, int64_t ntiles,
                                mxa_scale_mode mode, int views, int hadamard, mxa_qview* row, mxa_qview* tok,
                                cudaStream_t stream) {
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MXA_ERR_ARG;
  if (weight && !aligned(weight, 4)) return MXA_ERR_ALIGN;
  return quantize_impl(x, T, H, d, cu_seqlens, num_docs, max_seqlen, ntiles, mode, views, hadamard, row, tok, 1,
                       weight, eps, stream);
}

mxa_status mxa_quantize_key(const void* x, int64_t T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                            int max_seqlen, int64_t ntiles, mxa_qview* key, cudaStream_t stream) {
  if (!x || !key || T < 0 || T > 0x7FFFFFFFll || H <= 0 || H > 65535 || num_docs <= 0 || num_docs > 65535 ||
      ntiles <= 0 || max_seqlen <= 0)
    return MXA_ERR_ARG;
  if (d != 64 && d != 128) return MXA_ERR_UNSUPPORTED;
  if (!cu_seqlens && (T % num_docs != 0 || T / num_docs > max_seqlen)) return MXA_ERR_ARG;
  if (!aligned(x, 16)) return MXA_ERR_ALIGN;
  mxa_status st = check_view(*key);
  if (st != MXA_OK) return st;
  if (T == 0) return MXA_OK;
  if (cudaMemsetAsync(key->scales, 0x7F, mxa_key_scale_bytes(H, ntiles), stream) != cudaSuccess) return MXA_ERR_CUDA;
  KeyQuantArgs a{};
  a.x = x;
  a.T = T;
  a.H = H;
  a.cu_seqlens = cu_seqlens;
  a.num_docs = num_docs;
  a.ntiles = ntiles;
  a.codes = key->codes;
  a.scales = key->scales;
  const int maxlen = cu_seqlens ? max_seqlen : static_cast<int>(T / num_docs);
  if (launch_quantize_key(a, d, maxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;
  return MXA_OK;
}

size_t mxa_fwd_workspace_bytes(const mxa_fwd_params* p) {
  if (!p || check_shape(p->shape) != MXA_OK || !uses_list(p->shape)) return 0;
  return list_bytes(p->shape, q_side(p->shape));
}

mxa_status mxa_fwd(const mxa_fwd_params* p, cudaStream_t stream) {
  if (!p) return MXA_ERR_ARG;
  const mxa_shape& s = p->shape;
  mxa_status st = check_shape(s);
  if (st != MXA_OK) return st;
  if ((st = check_view(p->q_row)) != MXA_OK || (st = check_view(p->k_row)) != MXA_OK ||
      (st = check_view(p->v_tok)) != MXA_OK)
    return st;
  if (!p->o || !p->lse) return MXA_ERR_ARG;
  if (!aligned(p->o, 16) || !aligned(p->lse, 4)) return MXA_ERR_ALIGN;
  // strict causal fold on the diagonal tile (self-attention only)
  const bool fold = p->v_key.codes != nullptr;
  if (fold) {
    if ((st = check_view(p->v_key)) != MXA_OK) return st;
    if (is_cross(s)) return MXA_ERR_UNSUPPORTED;
  }
  const bool use_list = p->workspace && uses_list(s) && p->workspace_bytes >= list_bytes(s, q_side(s));
  if (use_list && !aligned(p->workspace, 256)) return MXA_ERR_ALIGN;
  if (s.T == 0) return MXA_OK;
  const Side qs = q_side(s), ks = k_side(s);
  FwdMaps maps;
  if (!make_code_map(&maps.q, p->q_row.codes, s.T, s.Hq, s.d) ||
      !make_code_map(&maps.k, p->k_row.codes, ks.T, s.Hkv, s.d) ||
      !make_code_map(&maps.v, p->v_tok.codes, ks.T, s.Hkv, s.d))
    return MXA_ERR_CUDA;
  if (fold && s.causal && !make_code_map(&maps.vkey, p->v_key.codes, ks.T, s.Hkv, s.d)) return MXA_ERR_CUDA;
  FwdArgs a{};
  a.T = s.T;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.cu_seqlens = s.cu_seqlens;
  a.num_docs = s.num_docs;
  a.ntiles = s.ntiles;
  set_k_side(a, s);
  a.causal = s.causal ? 1 : 0;
  a.alpha = alpha_of(s);
  a.scale_log2 = a.alpha * 1.4426950408889634f;
  a.q_sf = p->q_row.scales;
  a.k_sf = p->k_row.scales;
  a.v_sf = p->v_tok.scales;
  a.vkey_sf = (fold && s.causal) ? p->v_key.scales : nullptr;
  a.o = p->o;
  a.lse = p->lse;
  a.err = device_error_word();
  const int maxlen = max_len(s);
  if (use_list) {
    if (launch_tile_list(qs, ks, s.num_docs, a.causal, 0, p->workspace, stream) != cudaSuccess) return MXA_ERR_CUDA;
    a.items = tile_list_items(p->workspace);
    a.item_count = static_cast<const int32_t*>(p->workspace);
  }
  a.nq_tiles_doc = static_cast<int>((s.T / s.num_docs + 127) / 128);
  a.nk_tiles_doc = static_cast<int>((ks.T / s.num_docs + 127) / 128);
  if (launch_fwd(a, maps, s.d, maxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;
  return MXA_OK;
}

namespace {

// Backward workspace: padded D and LSE rows, the query and key tile lists, then
// either the dS blocks the dK/dV kernel emits for the dQ GEMM (both modes) or,
// in FP16 x 2^9 mode without room for them, the fp16 dQ accumulator of the
// fused kernel.
size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// FP16 per-row boost mode: the boost of every query row (fp32 [Hq, T]), the
// key bound of every (token, kv head) (int32 [T, Hkv]) and the per-tile key
// maxima (int32 [Hkv, NT]).
size_t bwd_boost_bytes(const mxa_shape& s, int dq_mode) {
  if (dq_mode != MXA_DQ_FP16_ROW || s.T <= 0) return 0;
  const size_t T = static_cast<size_t>(s.T);
  const size_t hkv = static_cast<size_t>(s.Hkv > 0 ? s.Hkv : 0);
  return round256(static_cast<size_t>(s.Hq) * T * 4) + round256(T * hkv * 4) +
         round256(hkv * static_cast<size_t>(s.ntiles > 0 ? s.ntiles : 0) * 4);
}

size_t bwd_head_bytes(const mxa_shape& s, int dq_mode = MXA_DQ_FP32) {
  return bwd_rows_bytes(s) + bwd_boost_bytes(s, dq_mode) + list_bytes(s, q_side(s)) + list_bytes(s, k_side(s));
}

size_t bwd_acc16_bytes(const mxa_shape& s) {
  const size_t b = static_cast<size_t>(s.T) * static_cast<size_t>(s.Hq) * static_cast<size_t>(s.d) * 2;
  return (b + 255) & ~size_t(255);
}

bool bwd_shape_sizable(const mxa_bwd_params* p) {
  return p && p->shape.T >= 0 && p->shape.Hq > 0 && (p->shape.d == 64 || p->shape.d == 128);
}

}  // namespace

size_t mxa_bwd_workspace_min_bytes(const mxa_bwd_params* p) {
  if (!bwd_shape_sizable(p)) return 0;
  const size_t head = bwd_head_bytes(p->shape, p->dq_mode);
  const bool strict = p->k_key.codes != nullptr;
  if (p->dq_mode == MXA_DQ_FP16_ROW || strict) return head + bwd_ds_bytes(p->shape, strict);  // the dQ GEMM only
  if (p->dq_mode != MXA_DQ_FP16_X512) return head;
  const size_t acc = bwd_acc16_bytes(p->shape), ds = bwd_ds_bytes(p->shape);
  return head + (acc < ds ? acc : ds);
}

size_t mxa_bwd_workspace_bytes(const mxa_bwd_params* p) {
  if (!bwd_shape_sizable(p)) return 0;
  return bwd_head_bytes(p->shape, p->dq_mode) + bwd_ds_bytes(p->shape, p->k_key.codes != nullptr);
}

mxa_status mxa_bwd(const mxa_bwd_params* p, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!p) return MXA_ERR_ARG;
  const mxa_shape& s = p->shape;
  mxa_status st = check_shape(s);
  if (st != MXA_OK) return st;
  const mxa_qview* vs[] = {&p->q_row, &p->k_row, &p->v_row, &p->g_row, &p->q_tok, &p->k_tok, &p->g_tok};
  for (const mxa_qview* v : vs)
    if ((st = check_view(*v)) != MXA_OK) return st;
  if (!p->o || !p->lse || !p->dq || !p->dk || !p->dv) return MXA_ERR_ARG;
  if (!aligned(p->o, 16) || !aligned(p->lse, 4) || !aligned(p->dq, 16) || !aligned(p->dk, 16) ||
      !aligned(p->dv, 16))
    return MXA_ERR_ALIGN;
  if (p->dq_mode != MXA_DQ_FP32 && p->dq_mode != MXA_DQ_FP16_X512 && p->dq_mode != MXA_DQ_FP16_ROW)
    return MXA_ERR_ARG;
  if (is_cross(s) && p->dq_mode != MXA_DQ_FP32) return MXA_ERR_UNSUPPORTED;
  const bool strict = p->k_key.codes != nullptr;  // strict dQ (the dQ GEMM path only)
  if (strict) {
    if ((st = check_view(p->k_key)) != MXA_OK) return st;
    if (is_cross(s)) return MXA_ERR_UNSUPPORTED;
  }
  if (!workspace || ws_bytes < mxa_bwd_workspace_min_bytes(p)) return MXA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MXA_ERR_ALIGN;
  if (s.T == 0) return MXA_OK;
  const Side qs = q_side(s), ks = k_side(s);
  BwdMaps maps;
  if (!make_code_map(&maps.q, p->q_row.codes, s.T, s.Hq, s.d) ||
      !make_code_map(&maps.k, p->k_row.codes, ks.T, s.Hkv, s.d) ||
      !make_code_map(&maps.v, p->v_row.codes, ks.T, s.Hkv, s.d) ||
      !make_code_map(&maps.g, p->g_row.codes, s.T, s.Hq, s.d) ||
      !make_code_map(&maps.qt, p->q_tok.codes, s.T, s.Hq, s.d) ||
      !make_code_map(&maps.kt, p->k_tok.codes, ks.T, s.Hkv, s.d) ||
      !make_code_map(&maps.gt, p->g_tok.codes, s.T, s.Hq, s.d))
    return MXA_ERR_CUDA;
  if (strict && !make_code_map(&maps.kkey, p->k_key.codes, ks.T, s.Hkv, s.d)) return MXA_ERR_CUDA;
  const size_t T = static_cast<size_t>(s.T), Hq = static_cast<size_t>(s.Hq), d = static_cast<size_t>(s.d);
  const size_t pad_elems = Hq * static_cast<size_t>(s.ntiles) * 128;
  const size_t dbytes = 2 * pad_elems * 4;
  float* dpad = static_cast<float*>(workspace);
  float* lpad = dpad + pad_elems;
  const bool rowboost = p->dq_mode == MXA_DQ_FP16_ROW;
  float* boost = rowboost ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + dbytes) : nullptr;
  int32_t* key_bound =
      rowboost ? reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(boost) + round256(Hq * T * 4)) : nullptr;
  void* qlist = static_cast<uint8_t*>(workspace) + dbytes + bwd_boost_bytes(s, p->dq_mode);
  void* klist = static_cast<uint8_t*>(qlist) + list_bytes(s, qs);
  void* acc = static_cast<uint8_t*>(klist) + list_bytes(s, ks);
  const bool fp16 = p->dq_mode != MXA_DQ_FP32;
  // dS emitted by the dK/dV kernel and summed by the dQ GEMM, else (FP32: dS
  // formed again by the dQ kernel; FP16: the fused kernel's fp16 accumulator)
  const bool emit = ws_bytes >= mxa_bwd_workspace_bytes(p);
  if (!emit && (strict || (fp16 && (rowboost || ws_bytes < bwd_head_bytes(s) + bwd_acc16_bytes(s)))))
    return MXA_ERR_WORKSPACE;
  const size_t acc_bytes = fp16 && !emit ? T * Hq * d * 2 : 0;
  const int maxlen = s.cu_seqlens ? s.max_seqlen : static_cast<int>(s.T / s.num_docs);

  PrepArgs pa{};
  pa.T = s.T;
  pa.Hq = s.Hq;
  pa.d = s.d;
  pa.g_codes = p->g_row.codes;
  pa.g_sf = p->g_row.scales;
  pa.cu_seqlens = s.cu_seqlens;
  pa.num_docs = s.num_docs;
  pa.ntiles = s.ntiles;
  pa.o = p->o;
  pa.lse = p->lse;
  pa.dpad = dpad;
  pa.lpad = lpad;
  pa.dq_acc = acc;
  pa.dq_acc_bytes = acc_bytes;
  pa.dq_boost = boost;
  pa.key_bound = key_bound;
  pa.Hkv = s.Hkv;
  pa.causal = s.causal ? 1 : 0;
  pa.alpha = alpha_of(s);
  if (rowboost) {
    KeyBoundArgs kb{};
    kb.T = s.T;
    kb.Hkv = s.Hkv;
    kb.d = s.d;
    kb.cu_seqlens = s.cu_seqlens;
    kb.num_docs = s.num_docs;
    kb.ntiles = s.ntiles;
    kb.causal = s.causal ? 1 : 0;
    kb.v_codes = p->v_row.codes;
    kb.v_sf = p->v_row.scales;
    kb.k_codes = p->k_row.codes;
    kb.k_sf = p->k_row.scales;
    kb.key_bound = key_bound;
    kb.tile_max = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(key_bound) +
                                             round256(T * static_cast<size_t>(s.Hkv) * 4));
    if (launch_key_bound(kb, maxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;
  }
  if (launch_bwd_prep(pa, maxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;

  BwdArgs a{};
  a.T = s.T;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.cu_seqlens = s.cu_seqlens;
  a.num_docs = s.num_docs;
  a.ntiles = s.ntiles;
  set_k_side(a, s);
  a.causal = s.causal ? 1 : 0;
  a.alpha = alpha_of(s);
  a.scale_log2 = a.alpha * 1.4426950408889634f;
  a.q_sf = p->q_row.scales;
  a.k_sf = p->k_row.scales;
  a.v_sf = p->v_row.scales;
  a.g_sf = p->g_row.scales;
  a.qt_sf = p->q_tok.scales;
  a.kt_sf = p->k_tok.scales;
  a.gt_sf = p->g_tok.scales;
  a.lpad = lpad;
  a.dpad = dpad;
  a.dq_mode = p->dq_mode;
  a.dq_acc32 = nullptr;
  a.dq_acc16 = acc_bytes ? static_cast<uint16_t*>(acc) : nullptr;
  a.dq_boost = boost;
  a.kkey_sf = strict ? p->k_key.scales : nullptr;
  a.dk = p->dk;
  a.dv = p->dv;
  a.dq_out = p->dq;
  a.err = device_error_word();
  a.mt = static_cast<int>(max_doc_tiles(s));
  if ((!fp16 || emit) && uses_list(s)) {
    if (launch_tile_list(qs, ks, s.num_docs, a.causal, 0, qlist, stream) != cudaSuccess ||
        launch_tile_list(ks, qs, s.num_docs, a.causal, 1, klist, stream) != cudaSuccess)
      return MXA_ERR_CUDA;
    a.q_items = tile_list_items(qlist);
    a.q_count = static_cast<const int32_t*>(qlist);
    a.k_items = tile_list_items(klist);
    a.k_count = static_cast<const int32_t*>(klist);
  }
  const int amaxlen = max_len(s);  // grids of the attention kernels
  // dK/dV kernel, then dQ summed in a fixed key-tile order (FP32 in TMEM, or
  // FP16 x 2^9 in registers) over the dS the dK/dV kernel emitted when the
  // workspace holds it; FP32 otherwise by a kernel that forms dS again
  if (!fp16 || emit) {
    if (emit) {
      a.ds_codes = static_cast<uint8_t*>(acc);
      a.ds_sf = a.ds_codes + static_cast<size_t>(s.Hq) * static_cast<size_t>(ks.ntiles) * a.mt * 16384;
      if (launch_bwd_emit(a, maps, s.d, amaxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;
      return MXA_OK;
    }
    if (launch_bwd_split(a, maps, s.d, amaxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;
    return MXA_OK;
  }
  if (launch_bwd(a, maps, s.d, maxlen, stream) != cudaSuccess) return MXA_ERR_CUDA;

  DqConvArgs c{};
  c.n = static_cast<int64_t>(T * Hq * d);
  c.acc32 = a.dq_acc32;
  c.acc16 = a.dq_acc16;
  c.mode = p->dq_mode;
  c.dq = p->dq;
  if (launch_dq_convert(c, stream) != cudaSuccess) return MXA_ERR_CUDA;
  return MXA_OK;
}

mxa_status mxa_get_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MXA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(int)) != cudaSuccess) return MXA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_err_word, &zero, sizeof(int));
    return MXA_ERR_TIMEOUT;
  }
  return MXA_OK;
}

}  // extern "C"
