// kernels.cuh -- kernel argument structs, shared device helpers and launchers.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxa {

// Bytes of one scale atom: 128 rows x 4 groups of 32, in the order the
// tensor core reads after a 32x128b.warpx4 copy: byte (r % 32) * 16 +
// (r / 32) * 4 + g.
constexpr int kAtomBytes = 512;

__device__ __forceinline__ int atom_offset(int r, int g) { return (r & 31) * 16 + (r >> 5) * 4 + g; }

// Document b: first token and length.  cu == nullptr: num_docs equal docs.
__device__ __forceinline__ void doc_bounds(const int32_t* cu, int num_docs, int64_t T, int b, int64_t& start,
                                           int64_t& len) {
  if (cu) {
    start = cu[b];
    len = static_cast<int64_t>(cu[b + 1]) - cu[b];
  } else {
    const int64_t L = T / num_docs;
    start = static_cast<int64_t>(b) * L;
    len = L;
  }
}

// One work item of a cost-sorted tile list: (document, 128-token tile of the
// list's side, first scale tile of the document on that side, first scale
// tile of the document on the other side).  A query list's items are query
// tiles (the other side: keys and values); a key list's items are key tiles.
struct alignas(16) TileItem {
  int32_t doc, tile, tile_base, other_base;
};
constexpr int kTileListHeader = 256;     // the item count, padded
constexpr int kTileListMaxCost = 4094;   // most tiles per document the list builder handles

// One side of an attention call: documents of `cu` (device offsets, or
// nullptr for num_docs equal documents of T / num_docs tokens).
struct Side {
  const int32_t* cu;
  int64_t T;
  int64_t ntiles;  // NT of its scale layouts
  int max_tiles;   // 128-token tiles of its longest document
};

// Bytes of one list over `ntiles` items of num_docs documents (256-byte multiple).
size_t tile_list_bytes(int num_docs, int64_t ntiles);
bool tile_lists_supported(int max_tiles);
// Build one list into ws (one CTA; stream-ordered): items are the tiles of
// `items`, ordered by the tiles of `other` each visits (longest first); with
// causal (self-attention only) a query tile t visits t + 1 key tiles
// (key_list = 0) and a key tile t feeds n_t - t query tiles (key_list = 1).
cudaError_t launch_tile_list(const Side& items, const Side& other, int num_docs, int causal, int key_list, void* ws,
                             cudaStream_t stream);
inline const TileItem* tile_list_items(const void* ws) {
  return reinterpret_cast<const TileItem*>(static_cast<const uint8_t*>(ws) + kTileListHeader);
}

struct QuantArgs {
  const void* x;  // bf16 [T, H, d]
  int64_t T;
  int H;
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;  // scale tiles NT (128-token tiles summed over documents)
  int write_row, write_tok;
  uint8_t* row_codes;
  uint8_t* row_scales;  // [H, NT, 512]
  uint8_t* tok_codes;
  uint8_t* tok_scales;  // [H, NT, 512]
  // RMSNorm prologue (rms != 0): every (token, head) vector becomes
  // x / sqrt(mean(x^2) + rms_eps) * rms_w before it is quantized
  int rms;
  const float* rms_w;  // fp32 [d] or null (all ones)
  float rms_eps;
};

// Per-key view: one UE8M0 exponent per (token, head) over all d channels.
struct KeyQuantArgs {
  const void* x;  // bf16 [T, H, d]
  int64_t T;
  int H;
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;
  uint8_t* codes;   // [T, H, d]
  uint8_t* scales;  // [H, NT, 128], tile-padded per document
};

struct FwdArgs {
  int64_t T;
  int Hq, Hkv;
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;
  // key/value side (the query side's own values for self-attention)
  int64_t Tk;
  const int32_t* cu_k;
  int64_t ntiles_k;
  int causal;
  float scale_log2;  // alpha * log2(e)
  float alpha;
  const uint8_t* q_sf;  // ROW scales of Q [Hq, NT, 512]
  const uint8_t* k_sf;  // ROW scales of K [Hkv, NT_k, 512]
  const uint8_t* v_sf;  // TOK scales of V [Hkv, NT_k, 512]
  // per-key view of V (null: no fold): UE8M0 exponent per key [Hkv, NT, 128];
  // its codes are read through FwdMaps::vkey on the causal diagonal tile
  const uint8_t* vkey_sf;
  void* o;              // bf16 [T, Hq, d]
  float* lse;           // [Hq, T]
  int* err;
  // cost-sorted query-tile list: item i / Hq for head i % Hq of virtual
  // item i.  With a list, or with equal documents on both sides (no
  // offsets), the launch is persistent: one CTA per virtual item, and each
  // running CTA takes over the items of CTAs not yet started (cluster launch
  // control); other calls take one CTA per (tile slot, document, head) of
  // the max_seqlen grid.
  const TileItem* items;
  const int32_t* item_count;
  int nq_tiles_doc, nk_tiles_doc;  // 128-token tiles per document (equal documents)
};

struct BwdArgs {
  int64_t T;
  int Hq, Hkv;
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;
  // key/value side (the query side's own values for self-attention)
  int64_t Tk;
  const int32_t* cu_k;
  int64_t ntiles_k;
  int causal;
  float scale_log2;
  float alpha;
  const uint8_t* q_sf;   // Q ROW
  const uint8_t* k_sf;   // K ROW
  const uint8_t* v_sf;   // V ROW
  const uint8_t* g_sf;   // G ROW
  const uint8_t* qt_sf;  // Q TOK
  const uint8_t* kt_sf;  // K TOK
  const uint8_t* gt_sf;  // G TOK
  const float* lpad;     // LSE * log2(e), tile-padded [Hq, NT, 128]; +inf on rows past a document's end
  const float* dpad;     // D, tile-padded [Hq, NT, 128]; 0 on rows past a document's end
  float* dq_acc32;       // [T, Hq, d] (FP32 mode)
  uint16_t* dq_acc16;    // [T, Hq, d] fp16 bits (FP16 x 2^9 mode)
  const float* dq_boost; // [Hq, T]: per-row boost 2^beta of the FP16 per-row mode (else null: 2^9)
  void* dk;              // bf16 [Tk, Hkv, d]
  void* dv;              // bf16 [Tk, Hkv, d]
  void* dq_out;          // bf16 [T, Hq, d] (written directly by the deterministic dQ kernel)
  // dS emitted by the dK/dV kernel for the dQ product (null: the dQ kernel
  // recomputes it).  Tile pair (h, document b, key tile kt, query tile qi)
  // has index ((h * NT_k + TBk_b + kt) * mt + qi): codes at 16 KB per pair, 128
  // key rows of 128 query bytes kept as their 128-byte-swizzled shared-memory
  // image (16-byte chunk c of row r at chunk c ^ (r % 8)); the 16 UE8M0 block
  // scales of a pair at 16 bytes per pair, byte 4 * (query block) + (key
  // block).
  uint8_t* ds_codes;
  uint8_t* ds_sf;
  // strict dQ (null: off): the per-key exponents of K [Hkv, NT, 128] (its
  // codes through BwdMaps::kkey).  The emitted dS then carries one scale per
  // (query row, 32 keys) -- a 512-byte atom per pair in the A-scale layout,
  // byte (q % 32) 16 + (q / 32) 4 + key block -- and on the diagonal pair
  // each key's dS column is folded with 2^e_k and multiplied with the
  // per-key K codes (scale 1)
  const uint8_t* kkey_sf;
  int mt;                // max 128-token query tiles of one document
  int dq_mode;
  int* err;
  // cost-sorted tile lists (null: max_seqlen grids); CTA i of the dK/dV
  // kernel takes key item i / Hkv for KV head i % Hkv, the dQ kernels query
  // item i / Hq for head i % Hq
  const TileItem* q_items;
  const int32_t* q_count;
  const TileItem* k_items;
  const int32_t* k_count;
};

struct PrepArgs {
  int64_t T;
  int Hq, d;
  const uint8_t* g_codes;  // G ROW codes [T, Hq, d]
  const uint8_t* g_sf;     // G ROW scales [Hq, NT, 512]
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;
  const void* o;     // bf16 [T, Hq, d]
  const float* lse;  // [Hq, T], the forward's LSE
  float* dpad;       // D, tile-padded [Hq, NT, 128]
  float* lpad;       // LSE * log2(e), tile-padded [Hq, NT, 128]
  void* dq_acc;      // zeroed here
  size_t dq_acc_bytes;
  // FP16 per-row boost mode (null otherwise): 2^beta of every query row,
  // from its G row, the key bound of its kv head and its visible key count
  float* dq_boost;           // [Hq, T]
  const int32_t* key_bound;  // [T, Hkv]: V + K exponent bound over the keys a row sees
  int Hkv;
  int causal;
  float alpha;
};

// Key bound of the FP16 per-row boost: for every (token t, kv head), the
// maxima over the keys that query t sees of cl2(max_c |V~_jc|) and of
// cl2(max_c |K~_jc|) (ROW views), summed.
struct KeyBoundArgs {
  int64_t T;
  int Hkv, d;
  const int32_t* cu_seqlens;
  int num_docs;
  int64_t ntiles;
  int causal;
  const uint8_t* v_codes;
  const uint8_t* v_sf;
  const uint8_t* k_codes;
  const uint8_t* k_sf;
  int32_t* key_bound;  // [T, Hkv]
  int32_t* tile_max;   // [Hkv, NT]: per 128-token tile, the maxima of v and k (int16 each)
};

struct DqConvArgs {
  int64_t n;  // elements
  const float* acc32;
  const uint16_t* acc16;
  int mode;
  void* dq;  // bf16
};

// Tensor maps of one attention call (3-D: d, H, T; SW128 for d = 128, SW64 for d = 64).
struct FwdMaps {
  CUtensorMap q, k, v, vkey;  // vkey: set only when FwdArgs::vkey_sf is
};
struct BwdMaps {
  CUtensorMap q, k, v, g, qt, kt, gt, kkey;  // kkey: set only when BwdArgs::kkey_sf is
};

cudaError_t launch_quantize_key(const KeyQuantArgs& a, int d, int max_seqlen, cudaStream_t stream);
cudaError_t launch_quantize(const QuantArgs& a, int d, bool tokblock, bool hadamard, int max_groups,
                            cudaStream_t stream);
cudaError_t launch_fwd(const FwdArgs& a, const FwdMaps& m, int d, int max_seqlen, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream);
cudaError_t launch_bwd_split(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream);
// dK/dV kernel emitting dS, then the dQ product over the emitted dS
cudaError_t launch_bwd_emit(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream);
cudaError_t launch_dq_gemm(const BwdArgs& a, const BwdMaps& m, int d, int max_seqlen, cudaStream_t stream);
cudaError_t launch_key_bound(const KeyBoundArgs& a, int max_seqlen, cudaStream_t stream);
cudaError_t launch_bwd_prep(const PrepArgs& a, int max_seqlen, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvArgs& a, cudaStream_t stream);

int* device_error_word();

}  // namespace mxa
