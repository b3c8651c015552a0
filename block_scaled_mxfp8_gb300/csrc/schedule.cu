// schedule.cu -- cost-sorted work lists of 128-token tiles for packed
// documents (one launch, one CTA per list).
//
// FLAMIA notes, Algorithm 2 (scheduling of jagged and causal work): every
// (document, tile) pair of one side becomes one work item, the items are
// ordered by the number of 128-token tiles of the other side they visit,
// largest first, and CTA i of an attention launch takes item i / H for head
// i % H.  The block scheduler hands out CTAs in index order, so the longest
// items start first (longest-processing-time order), the short ones fill the
// tail, and no CTA is launched for a tile slot past the end of a document.
//
// Lists:
//   query list (forward, dQ): items are query tiles; query tile t of a
//       document visits t + 1 key tiles when causal, else all n_k tiles of its
//       document's keys;
//   key list (dK/dV): items are key tiles; key tile t feeds n_t - t query
//       tiles when causal, else all n_q tiles of its document's queries.
// Causal masks exist for self-attention only (both sides the same).
// Items of equal cost keep no particular order (they are placed through
// shared-memory atomics); results do not depend on the order.
//
// Workspace layout of one list (kTileListHeader bytes of header, then the
// arrays): int32 count (number of items) at offset 0, TileItem items[NT of the
// item side], int32 base_items[num_docs] and base_other[num_docs] (first tile
// of each document on either side).
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

// Exclusive scan of per-document tile counts in chunks of the block; writes
// the first tile of every document and returns the total.
__device__ int scan_doc_tiles(const Side& sd, int num_docs, int* base, int* s_warp, int* s_carry) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t Lb = sd.cu ? 0 : sd.T / num_docs;
  if (tid == 0) *s_carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < num_docs; c0 += kThreads) {
    const int b = c0 + tid;
    int tiles = 0;
    if (b < num_docs) {
      const int64_t n = sd.cu ? static_cast<int64_t>(sd.cu[b + 1]) - sd.cu[b] : Lb;
      tiles = static_cast<int>((n + 127) / 128);
      if (tiles > sd.max_tiles) tiles = sd.max_tiles;  // the longest document bounds every one
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
    if (b < num_docs) base[b] = *s_carry + x - tiles + (warp > 0 ? s_warp[warp - 1] : 0);
    __syncthreads();
    if (tid == 0) *s_carry += s_warp[31];
    __syncthreads();
  }
  return *s_carry;
}

__global__ void __launch_bounds__(kThreads, 1)
    tile_list_kernel(const Side items, const Side other, int num_docs, int causal, int key_list, uint8_t* ws) {
  __shared__ int s_cur[kTileListMaxCost + 2];  // per cost: item count, then first slot, then a cursor
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x;
  int* count_out = reinterpret_cast<int*>(ws);
  TileItem* list = reinterpret_cast<TileItem*>(ws + kTileListHeader);
  int* base_i = reinterpret_cast<int*>(list + items.ntiles);
  int* base_o = base_i + num_docs;
  const int max_cost = causal ? items.max_tiles : other.max_tiles;
  const int nb = max_cost + 2;  // costs 0 .. max_cost + 1 (the last one only as a difference-array end)
  for (int i = tid; i < nb; i += kThreads) s_cur[i] = 0;

  // first tiles of every document on both sides
  const int total = scan_doc_tiles(items, num_docs, base_i, s_warp, &s_carry);
  const int total_o = scan_doc_tiles(other, num_docs, base_o, s_warp, &s_carry);

  // cost histogram: causal -- one item of each cost 1 .. n_t per document, as
  // a difference array; otherwise the n_t items of a document cost the
  // other side's tile count of that document
  for (int b = tid; b < num_docs; b += kThreads) {
    const int ti = (b + 1 < num_docs ? base_i[b + 1] : total) - base_i[b];
    if (ti <= 0) continue;
    if (causal) {
      atomicAdd(&s_cur[1], 1);
      atomicAdd(&s_cur[ti + 1], -1);
    } else {
      const int to = (b + 1 < num_docs ? base_o[b + 1] : total_o) - base_o[b];
      atomicAdd(&s_cur[to < max_cost ? to : max_cost], ti);
    }
  }
  __syncthreads();

  // items per cost, then the first slot of each cost in descending order:
  // first(c) = total - (items of cost at most c)
  if (causal) block_inclusive_scan(s_cur, nb, s_warp);
  block_inclusive_scan(s_cur, nb, s_warp);
  for (int i = tid; i < nb; i += kThreads) s_cur[i] = total - s_cur[i];
  __syncthreads();

  // place every item; its document by binary search on base_i
  for (int f = tid; f < total; f += kThreads) {
    int lo = 0, hi = num_docs;  // first document whose base exceeds f
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (base_i[mid] <= f) lo = mid + 1;
      else hi = mid;
    }
    const int b = lo - 1;
    const int base = base_i[b];
    const int ti = (b + 1 < num_docs ? base_i[b + 1] : total) - base;
    const int t = f - base;
    int cost;
    if (causal) {
      cost = key_list ? ti - t : t + 1;
    } else {
      const int to = (b + 1 < num_docs ? base_o[b + 1] : total_o) - base_o[b];
      cost = to < max_cost ? to : max_cost;
    }
    const int pos = atomicAdd(&s_cur[cost], 1);
    // an NT below the true tile count breaks the caller's contract (the
    // scale layouts are sized by it too); stay inside the list regardless
    if (pos < items.ntiles) list[pos] = TileItem{b, t, base, base_o[b]};
  }
  if (tid == 0) *count_out = total < items.ntiles ? total : static_cast<int>(items.ntiles);
}

}  // namespace

size_t tile_list_bytes(int num_docs, int64_t ntiles) {
  const size_t b = kTileListHeader + static_cast<size_t>(ntiles) * sizeof(TileItem) +
                   2 * static_cast<size_t>(num_docs) * sizeof(int32_t);
  return (b + 255) & ~size_t(255);
}

bool tile_lists_supported(int max_tiles) { return max_tiles >= 1 && max_tiles <= kTileListMaxCost; }

cudaError_t launch_tile_list(const Side& items, const Side& other, int num_docs, int causal, int key_list, void* ws,
                             cudaStream_t stream) {
  tile_list_kernel<<<1, kThreads, 0, stream>>>(items, other, num_docs, causal, key_list, static_cast<uint8_t*>(ws));
  return cudaGetLastError();
}

}  // namespace mxa
