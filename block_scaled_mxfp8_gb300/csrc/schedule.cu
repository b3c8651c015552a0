// schedule.cu -- cost-sorted work lists of 128-token tiles for packed
// documents (one launch, one CTA).
//
// FLAMIA notes, Algorithm 2 (scheduling of jagged and causal work): every
// (document, tile) pair becomes one work item, the items are ordered by the
// number of 128-key tiles they visit, largest first, and CTA i of an attention
// launch takes item i / H for head i % H.  The block scheduler hands out CTAs
// in index order, so the longest items start first (longest-processing-time
// order), the short ones fill the tail, and no CTA is launched for a tile slot
// past the end of a document.
//
// Two lists are written, both over the same items:
//   query list (forward, dQ): query tile t of a document with n_t tiles
//       visits t + 1 key tiles when causal, else n_t;
//   key list (dK/dV): key tile t visits n_t - t query tiles when causal,
//       else n_t.
// Items of equal cost keep no particular order (they are placed through
// shared-memory atomics); results do not depend on the order.
//
// Workspace layout (kTileListHeader bytes of header, then the arrays):
//   int32 count (number of items = sum of tiles) at offset 0,
//   TileItem q[NT], TileItem k[NT], int32 doc_base[num_docs] (first tile of
//   each document).
#include "kernels.cuh"

namespace mxa {

namespace {

constexpr int kThreads = 1024;

// Inclusive prefix sum of v[0, n) in shared memory, by the whole block.
__device__ void block_inclusive_scan(int* v, int n, int* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (int c0 = 0; c0 < n; c0 += kThreads) {
    const int i = c0 + tid;
    int x = i < n ? v[i] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    x += carry + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (i < n) v[i] = x;
    carry += warp_sums[31];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    tile_lists_kernel(const int32_t* cu, int num_docs, int64_t T, int causal, int max_tiles, int64_t ntiles,
                      uint8_t* ws) {
  __shared__ int s_cur_q[kTileListMaxCost + 2];  // per cost: item count, then first slot, then a cursor
  __shared__ int s_cur_k[kTileListMaxCost + 2];
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* count_out = reinterpret_cast<int*>(ws);
  TileItem* qlist = reinterpret_cast<TileItem*>(ws + kTileListHeader);
  TileItem* klist = qlist + ntiles;
  int* doc_base = reinterpret_cast<int*>(klist + ntiles);
  const int nb = max_tiles + 2;  // costs 0 .. max_tiles + 1 (the last one only as a difference-array end)
  for (int i = tid; i < nb; i += kThreads) s_cur_q[i] = 0;
  if (tid == 0) s_carry = 0;
  __syncthreads();

  // pass 1: first tile of every document (exclusive scan of the tile counts)
  // and the cost histogram (causal: one item of each cost 1 .. n_t per
  // document, kept as a difference array; otherwise n_t items of cost n_t;
  // the query and key lists have the same histogram)
  const int64_t Lb = cu ? 0 : T / num_docs;
  for (int c0 = 0; c0 < num_docs; c0 += kThreads) {
    const int b = c0 + tid;
    int tiles = 0;
    if (b < num_docs) {
      const int64_t n = cu ? static_cast<int64_t>(cu[b + 1]) - cu[b] : Lb;
      tiles = static_cast<int>((n + 127) / 128);
      if (tiles > max_tiles) tiles = max_tiles;  // max_seqlen bounds every document
    }
    int x = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int v = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      s_warp[lane] = v;
    }
    __syncthreads();
    if (b < num_docs) {
      doc_base[b] = s_carry + x - tiles + (warp > 0 ? s_warp[warp - 1] : 0);
      if (tiles > 0) {
        if (causal) {
          atomicAdd(&s_cur_q[1], 1);
          atomicAdd(&s_cur_q[tiles + 1], -1);
        } else {
          atomicAdd(&s_cur_q[tiles], tiles);
        }
      }
    }
    __syncthreads();
    if (tid == 0) s_carry += s_warp[31];
    __syncthreads();
  }
  const int total = s_carry;

  // items per cost, then the first slot of each cost in descending order:
  // first(c) = total - (items of cost at most c)
  if (causal) block_inclusive_scan(s_cur_q, nb, s_warp);
  block_inclusive_scan(s_cur_q, nb, s_warp);
  for (int i = tid; i < nb; i += kThreads) {
    const int first = total - s_cur_q[i];
    s_cur_q[i] = first;
    s_cur_k[i] = first;
  }
  __syncthreads();

  // pass 2: place every item; its document by binary search on doc_base
  for (int f = tid; f < total; f += kThreads) {
    int lo = 0, hi = num_docs;  // first document whose base exceeds f
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (doc_base[mid] <= f) lo = mid + 1;
      else hi = mid;
    }
    const int b = lo - 1;
    const int base = doc_base[b];
    const int tiles = (b + 1 < num_docs ? doc_base[b + 1] : total) - base;
    const int t = f - base;
    const int qcost = causal ? t + 1 : tiles;
    const int kcost = causal ? tiles - t : tiles;
    const int qpos = atomicAdd(&s_cur_q[qcost], 1);
    const int kpos = atomicAdd(&s_cur_k[kcost], 1);
    // an NT below the true tile count breaks the caller's contract (the
    // scale layouts are sized by it too); stay inside the lists regardless
    if (qpos < ntiles) qlist[qpos] = TileItem{b, t, base, qcost};
    if (kpos < ntiles) klist[kpos] = TileItem{b, t, base, kcost};
  }
  if (tid == 0) *count_out = total < ntiles ? total : static_cast<int>(ntiles);
}

}  // namespace

size_t tile_list_bytes(int num_docs, int64_t ntiles) {
  const size_t b = kTileListHeader + 2 * static_cast<size_t>(ntiles) * sizeof(TileItem) +
                   static_cast<size_t>(num_docs) * sizeof(int32_t);
  return (b + 255) & ~size_t(255);
}

bool tile_lists_supported(int max_tiles) { return max_tiles >= 1 && max_tiles <= kTileListMaxCost; }

cudaError_t launch_tile_lists(const int32_t* cu, int num_docs, int64_t T, int causal, int max_tiles, int64_t ntiles,
                              void* ws, cudaStream_t stream) {
  tile_lists_kernel<<<1, kThreads, 0, stream>>>(cu, num_docs, T, causal, max_tiles, ntiles,
                                                static_cast<uint8_t*>(ws));
  return cudaGetLastError();
}

}  // namespace mxa
