/*
 * mxa.h -- C ABI of libmxa.so: MXFP8 block-scaled attention (forward and
 * backward) for NVIDIA GB300 (sm_103a).
 *
 * What it computes (page titles and sections of the sources):
 *   - MXFP8 operands: E4M3 codes plus one UE8M0 power-of-two scale per 32
 *     values ("Flash Attention 4 + MXFP8 on Blackwell", "Что такое MXFP8";
 *     FLAMIA reading notes sec. 2 "两种硬件格式"), with the scale exponent
 *     e = ceil(log2(amax / 448)) (FLAMIA notes sec. 4, the saturation bound).
 *   - Attention S = alpha Q K^T, softmax over the visible keys, O = P V,
 *     LSE = m + ln l; backward dV = P^T G, dP = G V^T, D = G . O,
 *     dS = P (dP - D), dQ = alpha dS K, dK = alpha dS^T Q (FLAMIA notes
 *     sec. 2 and Algorithm 1).
 *   - P quantised online with a fixed boost 2^4 (2^8 for the backward dV
 *     product) (FLAMIA notes sec. 5 "概率上限由两个参数共同决定"); dS quantised
 *     in 32 x 32 blocks from the block max-abs, taken in the register layout
 *     without a transpose (FA4 write-up "Квантование dS без транспонирования").
 *   - dQ accumulated in FP32, in FP16 with a 2^9 boost (FA4 write-up, same
 *     section) or in FP16 with a per-row boost from the row's own bound
 *     (FLAMIA notes sec. 4, the strict accumulator scale).
 *   - Strict causal mode (FLAMIA notes sec. 4, moving the scale across the
 *     boundary): per-key views of V and K folded into P and dS on each
 *     query's diagonal tile, and per-query dS scales for the dQ product, so
 *     that no output of a row depends on a later position.
 *   - Cross-attention with separate key/value documents, cost-sorted tile
 *     work lists for packed documents (FLAMIA notes, Algorithm 2) and a fused
 *     RMSNorm + quantize producer (FA4 write-up).
 *   - Packed documents through cu_seqlens; scale groups never cross a
 *     document and only the scale tensors are padded ("Jagged-модуль без
 *     gather"; FLAMIA notes sec. 6).
 *   - Token-block mode: one exponent per 32 document-relative tokens x d of a
 *     head, the same codes serving both contraction axes, optional normalized
 *     128-point Hadamard rotation of Q/K (FLAMIA notes sec. 3).
 *
 * Conventions
 *   Tensors are token-major "THD": element (t, h, c) of a [T, H, d] tensor
 *   sits at offset (t * H + h) * d + c.  d is 64 or 128.
 *   Device pointers everywhere except where a parameter says "host".
 *   Ownership: the caller owns every buffer, including the backward workspace;
 *   the library never allocates device memory, never synchronizes a stream
 *   (except mxa_get_error) and keeps no pointer after a call returns.
 *   Asynchrony: calls are stream-ordered on the given cudaStream_t.
 *   Errors: argument errors return a status synchronously and launch
 *   nothing.  MXA_ERR_CUDA wraps a launch error.  A kernel whose internal wait
 *   runs out of time (it never spins forever) records an error word that
 *   mxa_get_error() reports as MXA_ERR_TIMEOUT.
 *   Inputs must be finite; non-finite inputs give unspecified codes.
 *
 * Scale layouts (UE8M0 bytes; 0x7F = 1.0 fills every unused byte)
 *   Both views store scales in 512-byte "atoms" that the tensor core consumes
 *   directly (a 128 x 4 block of scales: 128 rows of the MMA operand, 4
 *   groups of 32 along its contraction axis).  Inside an atom the scale of
 *   row r, group g sits at byte (r % 32) * 16 + (r / 32) * 4 + g.
 *   Each document b owns ceil(n_b / 128) consecutive atoms per head, one per
 *   128-token tile counted from the document start; its first atom index is
 *   TB_b = sum_{b' < b} ceil(n_b' / 128).  NT = TB_{num_docs} is the number of
 *   scale tiles (mxa_scale_tiles); a scale buffer holds H * NT atoms:
 *   atom (h, b, i) at byte offset ((h * NT + TB_b + i) * 512).
 *   ROW view (groups of 32 channels of one token and head): in atom
 *     (h, b, i), row r = the token at document position 128 i + r, group g =
 *     channels [32 g, 32 g + 32).
 *   TOK view (groups of 32 document-relative tokens of one head and
 *     channel): in atom (h, b, i), row r = channel r (d <= 128), group g =
 *     document positions [128 i + 32 g, 128 i + 32 g + 32); the last group of
 *     a document may be short; groups never cross a document.
 *   Only the scales are padded per document; codes stay at their packed
 *   token offsets.  In MXA_SCALE_TOKBLOCK32 mode the one exponent of each
 *   (document, 32-token block, head) is written into both layouts, and both
 *   views share one code buffer.
 */
#ifndef MXA_H
#define MXA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXA_ABI_VERSION 4

typedef enum {
  MXA_OK = 0,
  MXA_ERR_ARG = 1,         /* null pointer, bad size or flag */
  MXA_ERR_ALIGN = 2,       /* code buffer not 16-byte aligned, or scale buffer not 16-byte aligned */
  MXA_ERR_UNSUPPORTED = 3, /* d not in {64, 128}; Hadamard with d != 128; Hq % Hkv != 0 */
  MXA_ERR_WORKSPACE = 4,   /* backward workspace too small */
  MXA_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed */
  MXA_ERR_TIMEOUT = 6      /* a kernel gave up waiting (reported by mxa_get_error) */
} mxa_status;

typedef enum {
  MXA_SCALE_MX32 = 0,      /* 1-D groups of 32 along the contraction axis (row and token views) */
  MXA_SCALE_TOKBLOCK32 = 1 /* one exponent per 32 document-relative tokens x d, one code set */
} mxa_scale_mode;

enum { MXA_VIEW_ROW = 1, MXA_VIEW_TOK = 2 };

typedef enum {
  MXA_DQ_FP32 = 0,     /* dQ summed in fp32 over the key tiles, in a fixed order (deterministic; a
                          separate dQ kernel recomputes S and dP per query tile) */
  MXA_DQ_FP16_X512 = 1 /* dQ partial product of each 128-key tile boosted by 2^9, rounded to
                          fp16 and added into an fp16 sum, unboosted at the end: in key-tile
                          order in the dQ GEMM when the workspace holds the emitted dS
                          (deterministic), else with atomics in a fused kernel (order varies) */,
  MXA_DQ_FP16_ROW = 2  /* as FP16_X512 in the dQ GEMM, with a boost 2^beta_i per query row and
                          head instead of 2^9, chosen from magnitudes that query row i may
                          depend on -- its own G row and the maxima of V and K over the keys it
                          sees -- so no later position changes its rounding (FLAMIA notes sec.
                          4, the strict accumulator scale).  With the E4M3 decoding x~ of the
                          ROW views and cl2(x) = ceil(log2 x) (exact, on the scale exponents and
                          code bits):
                            beta_i = clamp(11 - cl2(alpha) - log2(d) - s(n_i) - g_i - V_i - K_i,
                                           -100, 100)
                            g_i = cl2(max_c |G~_ic|); V_i, K_i = max over the keys j that row i
                            sees (j <= i when causal, else the document) of cl2(max_c |V~_jc|),
                            cl2(max_c |K~_jc|); n_i = number of those keys;
                            s(n) = 1 + max(0, cl2(n) - 14).
                          Then 2^(15 - beta_i) bounds |dQ_i| and every partial sum of it, so
                          the fp16 sum cannot overflow: |dP_ij| <= d |G~_i| |V~_j| (max-abs
                          norms); O_i averages token-view V values, each within 32/15 of the
                          ROW view's maximum, so |D_i| <= 2.2 d |G~_i| V*; the E4M3 dS is
                          within 2x of dS; sum_j P_ij <= 16/15 + n_i 2^-14 <= 2^s(n_i) (weights
                          below the E4M3 range drop out of the forward's row sum); the
                          token-view K is within 32/15 of K*: |dQ_ic| <= alpha 2 (3.2 d
                          |G~_i| V*) 2^s (32/15) K* < 2^(4 + cl2(alpha) + log2 d + s + g + V + K).
                          An all-zero operand counts as cl2 = -2000 (beta = 100).  Needs the
                          full mxa_bwd_workspace_bytes(); self-attention only. */
} mxa_dq_mode;

/* One quantized view of a tensor: E4M3 codes [T, H, d] and its UE8M0 scales
 * in the layout of the view (see above).  Device pointers. */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
} mxa_qview;

/* ABI version (MXA_ABI_VERSION of the built library). */
int mxa_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* mxa_status_str(mxa_status s);

/* Number of scale tiles NT = sum over documents of ceil(n_b / 128).
 * cu_seqlens_host: host copy of the [num_docs + 1] offsets, or NULL for
 * num_docs equal documents of T / num_docs tokens.  Returns -1 on bad input. */
int64_t mxa_scale_tiles(int64_t T, int num_docs, const int32_t* cu_seqlens_host);

/* Upper bound on NT that needs no host copy of cu_seqlens:
 * ceil(T / 128) + num_docs. */
int64_t mxa_scale_tiles_bound(int64_t T, int num_docs);

/* Bytes of the scale buffer of one view (either layout): H * NT * 512. */
size_t mxa_scale_bytes(int H, int64_t ntiles);

/* Quantize a bf16 tensor x [T, H, d] into MXFP8 views.
 *   cu_seqlens: device int32 [num_docs + 1] document offsets, or NULL for
 *     num_docs equal documents (T % num_docs == 0).  max_seqlen bounds every
 *     document length (it sizes the grid).
 *   ntiles: NT of the scale layouts (mxa_scale_tiles or _bound); the same
 *     value must be given to mxa_fwd / mxa_bwd.
 *   mode: MXA_SCALE_MX32 -> `views` selects MXA_VIEW_ROW and/or MXA_VIEW_TOK;
 *     each selected view gets its own codes and scales.
 *     MXA_SCALE_TOKBLOCK32 -> one exponent per (document, 32-token block,
 *     head); views must be both; codes go to row->codes (tok->codes must be
 *     NULL or equal to it) and the exponent is written into both layouts.
 *   hadamard: first rotate every (token, head) vector by the normalized
 *     128-point Hadamard matrix (TOKBLOCK32 only, d == 128), in fp32, in the
 *     Sylvester butterfly order, then multiply by fp32(128^-1/2).
 *   Scale buffers are first filled with 0x7F (stream-ordered memset).
 *   Code buffers must be 16-byte aligned; scale buffers 16-byte aligned.
 * Status: MXA_OK, MXA_ERR_ARG, MXA_ERR_ALIGN, MXA_ERR_UNSUPPORTED,
 * MXA_ERR_CUDA. */
mxa_status mxa_quantize(const void* x_bf16, int64_t T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                        int max_seqlen, int64_t ntiles, mxa_scale_mode mode, int views, int hadamard,
                        mxa_qview* row, mxa_qview* tok, cudaStream_t stream);

/* Fused RMSNorm + quantize (FA4 write-up, "Fused RMSNorm+Quantize": the
 * normalization becomes the prologue of the pass that reads the data anyway,
 * instead of a pass of its own).  Every (token, head) vector of x is
 * normalized in IEEE fp32,
 *   y = x * (1 / sqrt(mean(x^2) + eps)) * weight,
 * and y (never rounded to bf16) is quantized exactly as mxa_quantize
 * quantizes x, into the same views, layouts and modes (the Hadamard rotation,
 * when asked for, applies to y).  The fp32 order is fixed: per 16-channel
 * chunk the squares summed in channel order, the chunk sums added pairwise,
 * correctly rounded sqrt and division; an all-zero vector with eps = 0 gives
 * y = 0.
 *   weight: device fp32 [d], or NULL for all ones; eps >= 0.
 * Status: as mxa_quantize, plus MXA_ERR_ARG for a negative or non-finite eps
 * and MXA_ERR_ALIGN for a weight not 4-byte aligned. */
mxa_status mxa_rmsnorm_quantize(const void* x_bf16, const float* weight, float eps, int64_t T, int H, int d,
                                const int32_t* cu_seqlens, int num_docs, int max_seqlen, int64_t ntiles,
                                mxa_scale_mode mode, int views, int hadamard, mxa_qview* row, mxa_qview* tok,
                                cudaStream_t stream);

/* Bytes of the scale buffer of a per-key view: H * NT * 128. */
size_t mxa_key_scale_bytes(int H, int64_t ntiles);

/* Per-key view of V for the strict causal forward (FLAMIA notes sec. 4,
 * moving the scale across the boundary: on the diagonal tile each key gets
 * its own power-of-two scale, which is folded into the probability operand,
 * P_ij (s_j v_j) = (P_ij s_j) v_j, so that no key's representation depends on
 * a later key of its 32-token group).  For every (token t, head h): e_t by
 * the MX rule over all d channels, e = ceil(log2(amax / 448)) (0 for an
 * all-zero vector), codes E4M3(x * 2^-e_t) (round to nearest even,
 * saturating).
 *   key->codes: [T, H, d], 16-byte aligned;
 *   key->scales: UE8M0 bytes [H, NT, 128], 16-byte aligned, tile-padded per
 *     document like the other scale layouts (byte (h NT + TB_b + t / 128) 128
 *     + t % 128 for document-relative token t of document b whose first tile
 *     is TB_b); first filled with 0x7F (stream-ordered memset).
 * Other arguments and the status codes as mxa_quantize. */
mxa_status mxa_quantize_key(const void* x_bf16, int64_t T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                            int max_seqlen, int64_t ntiles, mxa_qview* key, cudaStream_t stream);

/* Shape shared by the forward and backward calls.
 * Self-attention (T_k = 0): queries, keys and values share one token layout
 * (T, cu_seqlens, max_seqlen, ntiles).
 * Cross-attention (T_k > 0): the queries of document b attend to that
 * document's own keys and values, laid out by T_k, cu_seqlens_k, max_seqlen_k
 * and ntiles_k (the K and V views are quantized with those); Lq != Lk per
 * document, e.g. a few hundred query tokens against thousands of jagged
 * key/value tokens.  No causal mask (causal must be 0), FP32 dQ mode only,
 * and every document with queries must have at least one key. */
typedef struct {
  int64_t T;                  /* total query tokens */
  int Hq, Hkv, d;             /* query heads, key/value heads (Hq % Hkv == 0), head dim (64 or 128) */
  const int32_t* cu_seqlens;  /* device int32 [num_docs + 1], or NULL: num_docs equal documents */
  int num_docs;
  int max_seqlen;             /* longest document (grid size); must bound every document */
  int64_t ntiles;             /* NT of the scale layouts used when the views were quantized */
  int causal;                 /* 1: query i sees keys [doc start, i]; 0: the whole document */
  float softmax_scale;        /* alpha; 0 selects 1/sqrt(d) */
  int64_t T_k;                /* 0: self-attention; else total key/value tokens */
  const int32_t* cu_seqlens_k;  /* device int32 [num_docs + 1] of the keys, or NULL: equal documents */
  int max_seqlen_k;           /* longest key/value document */
  int64_t ntiles_k;           /* NT of the K and V scale layouts */
} mxa_shape;

typedef struct {
  mxa_shape shape;
  mxa_qview q_row;  /* Q, ROW view (scores) */
  mxa_qview k_row;  /* K, ROW view (scores) */
  mxa_qview v_tok;  /* V, TOK view (P V) */
  void* o;          /* out: bf16 [T, Hq, d] */
  float* lse;       /* out: fp32 [Hq, T], natural-log LSE (alpha included) */
  void* workspace;  /* optional device buffer (256-byte aligned) for the tile work list, or NULL */
  size_t workspace_bytes;
  mxa_qview v_key;  /* optional V per-key view (mxa_quantize_key), causal self-attention only:
                       with codes != NULL the P V product of every query's diagonal 128-key
                       tile uses it, with each key's scale folded into P (P'_ij = P_ij 2^e_j,
                       quantized per query row and 32 keys by the MX rule), so that O_i and
                       LSE_i depend on no key after i (FLAMIA notes sec. 4).  Other key tiles
                       are fully visible and keep v_tok.  NULL codes: no fold. */
} mxa_fwd_params;

/* Workspace bytes that let mxa_fwd take its CTAs from a cost-sorted work
 * list of packed documents (FLAMIA notes, Algorithm 2): one item per
 * (document, 128-query tile), so that no CTA is launched for a tile slot past
 * a document's end, ordered by the number of key tiles it visits, longest
 * first (item i / Hq for head i % Hq).  256 + 16 * ntiles + 8 * num_docs
 * bytes, rounded up to 256.  Returns 0 when the list brings nothing (equal
 * documents on both sides: cu_seqlens and cu_seqlens_k NULL) or cannot be
 * built (a side's longest document above 4094 tiles); with workspace NULL or
 * smaller, mxa_fwd launches one CTA per (tile slot of max_seqlen, document,
 * head).  Every call rebuilds the list on the device (cu_seqlens stays
 * device-only).  With a list, and on equal documents, the forward is
 * persistent: the grid holds one CTA per item and each running CTA takes
 * over the items of CTAs that have not started (cluster launch control), so
 * the longest items start first and the short ones fill in as CTAs free up
 * (strict mode on equal documents keeps one CTA per tile). */
size_t mxa_fwd_workspace_bytes(const mxa_fwd_params* p);

/* Forward: O = softmax(alpha Q K^T) V over the visible keys, and LSE.
 * Status: MXA_OK, MXA_ERR_ARG, MXA_ERR_ALIGN, MXA_ERR_UNSUPPORTED,
 * MXA_ERR_CUDA. */
mxa_status mxa_fwd(const mxa_fwd_params* p, cudaStream_t stream);

typedef struct {
  mxa_shape shape;
  mxa_qview q_row, k_row;  /* score views (rebuild S exactly as the forward did) */
  mxa_qview v_row, g_row;  /* dP = G V^T and D = G . O (the same G in both) */
  mxa_qview q_tok;         /* dK = alpha dS^T Q */
  mxa_qview k_tok;         /* dQ = alpha dS K */
  mxa_qview g_tok;         /* dV = P^T G */
  /* (for cross-attention k_row, v_row, k_tok are the key/value side's views) */
  const void* o;           /* bf16 [T, Hq, d], the forward's output */
  const float* lse;        /* fp32 [Hq, T], the forward's LSE */
  void* dq;                /* out: bf16 [T, Hq, d] */
  void* dk;                /* out: bf16 [T (T_k for cross-attention), Hkv, d], summed over the query heads of the group */
  void* dv;                /* out: bf16 [T (T_k for cross-attention), Hkv, d] */
  mxa_dq_mode dq_mode;
  mxa_qview k_key;         /* optional per-key view of K (mxa_quantize_key), self-attention only:
                              with codes != NULL dQ_i depends on no position after i (FLAMIA
                              notes sec. 4) -- the dS operand of the dQ product is quantized
                              with one scale per (query row, 32 keys) instead of per 32 x 32
                              block, and on each query's diagonal 128-key tile every key's dS
                              column is folded with its 2^e_k and multiplied with its per-key
                              codes (scale 1).  With the forward's v_key fold (so that O_i and
                              LSE_i are strict too), rows i <= p keep dQ_i bit for bit when
                              anything after p changes, G rows <= p fixed.  Needs the full
                              mxa_bwd_workspace_bytes(); dK and dV are unchanged (they depend
                              on later queries by definition).  NULL codes: off. */
} mxa_bwd_params;

/* Workspace bytes of mxa_bwd's fastest path.
 *   Both modes: D and LSE * log2(e), fp32, each padded to whole 128-token
 *   tiles per document ([Hq, ntiles, 128]); then the key-tile and query-tile
 *   work lists that schedule the dK/dV and dQ CTAs of packed documents as
 *   mxa_fwd schedules its own (for each of the query and the key side:
 *   256 + 16 * NT of that side + 8 * num_docs bytes, rounded up to 256;
 *   reserved in every case).
 *   Then the dS blocks the dK/dV pass emits for the dQ product --
 *   E4M3 codes (16 KB) and the 16 UE8M0 block scales per (query head, key
 *   tile, query tile of the same document) pair, with mt = ceil(max_seqlen /
 *   128) query-tile slots per key tile: Hq * NT_k * mt * 16400 bytes, NT_k
 *   the key side's ntiles (B8 H32 L4096: 4.3 GB).  With k_key (strict dQ) each pair
 *   carries a 512-byte scale atom instead of the 16 block scales (one UE8M0 per
 *   query row and key block, byte (q % 32) 16 + (q / 32) 4 + key block):
 *   Hq * NT_k * mt * (16384 + 512) bytes.
 *   FP16_ROW mode: after the D and LSE rows, before the lists, the boost
 *   2^beta_i of every query row as fp32 [Hq, T], the key bound V_t + K_t
 *   of every (token, kv head) as int32 [T, Hkv] and per-tile key maxima as
 *   int32 [Hkv, ntiles], each rounded up to 256 bytes. */
size_t mxa_bwd_workspace_bytes(const mxa_bwd_params* p);

/* Smallest workspace mxa_bwd accepts: the padded D and LSE rows and the tile
 * lists; in FP16_X512 mode plus the smaller of the emitted dS blocks and the
 * fp16 dQ accumulator [T, Hq, d] (rounded up to 256 bytes).  A workspace
 * smaller than mxa_bwd_workspace_bytes() selects, in FP32 mode, a dQ kernel
 * that forms dS again from S and dP instead of reading the emitted blocks
 * (slower; same blocks, so the same tolerances), and in FP16_X512 mode a fused
 * kernel that adds the boosted partials into the fp16 accumulator with
 * atomics (slower, order varies). */
size_t mxa_bwd_workspace_min_bytes(const mxa_bwd_params* p);

/* Backward.  workspace: device buffer of ws_bytes >= mxa_bwd_workspace_min_bytes()
 * bytes (mxa_bwd_workspace_bytes() for the fastest path), 256-byte aligned;
 * its contents on entry do not matter.
 * Status: MXA_OK, MXA_ERR_ARG, MXA_ERR_ALIGN, MXA_ERR_UNSUPPORTED,
 * MXA_ERR_WORKSPACE, MXA_ERR_CUDA. */
mxa_status mxa_bwd(const mxa_bwd_params* p, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Size of the library-owned scratch array that mxa_bwd_noalloc uses in place
 * of a caller workspace: 32 MiB on every GPU that loads the library. */
#define MXA_BWD_NOALLOC_MAX_WORKSPACE (32u * 1024u * 1024u)

/* Backward without a caller workspace.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory --
 * for instance code running under a framework whose caching allocator owns
 * all device memory and offers no side buffers, or a plugin host that gives
 * the library a fixed memory budget -- and therefore cannot provide
 * mxa_bwd's workspace.
 * Same arguments, results and status codes as mxa_bwd, computed the same way;
 * the workspace is a file-scope device array of MXA_BWD_NOALLOC_MAX_WORKSPACE
 * bytes that the library owns (held on every GPU that loads the library until
 * the process exits).  A call whose mxa_bwd_workspace_min_bytes() exceeds it
 * gets mxa_bwd's own argument checks and then MXA_ERR_WORKSPACE, with no
 * work launched.  FP32-mode calls need the D and LSE rows (2 * Hq * ntiles *
 * 512 bytes) plus, for packed or cross-attention inputs, the tile lists (16
 * bytes per scale tile and side, plus 256): B8 H32 L4096 needs 8 MiB; they
 * take the fast dQ path only when their full mxa_bwd_workspace_bytes() also
 * fits, else they form dS again in the dQ kernel.  The FP16 modes and the
 * strict dQ operand (k_key) also need the emitted dS or the fp16 dQ
 * accumulator, so only small calls fit.
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, which allocates nothing); the first call on a
 * device also loads the library's kernels there, so make it before any
 * stream capture.  The function allocates nothing.  Every call on a device
 * shares the one array and it keeps the last call's contents (each call
 * rewrites what it reads); calls that overlap on the GPU -- on different
 * streams, or from several threads -- race on it and must be serialized by
 * the caller. */
mxa_status mxa_bwd_noalloc(const mxa_bwd_params* p, cudaStream_t stream);

/* Synchronize `stream`, then report and clear the device error word of the
 * current device: MXA_OK, MXA_ERR_TIMEOUT (a kernel gave up waiting) or
 * MXA_ERR_CUDA. */
mxa_status mxa_get_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MXA_H */
