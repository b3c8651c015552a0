// noalloc.cu -- mxa_bwd_noalloc: the backward pass with its scratch space in a
// device array that the library itself owns, for callers that cannot allocate
// device memory (see include/mxa.h).  This file adds one entry point and
// changes no existing code path: it resolves the array's device address and
// hands it to mxa_bwd as the workspace.
#include "../../include/mxa.h"
#include "kernels.cuh"

namespace mxa {
namespace {

static_assert(MXA_BWD_NOALLOC_MAX_WORKSPACE % 256 == 0, "scratch size must keep 256-byte alignment");

// Scratch of mxa_bwd_noalloc.  A file-scope device array: every GPU that
// loads this library holds it until the process exits.  In host code its
// name is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[MXA_BWD_NOALLOC_MAX_WORKSPACE];

}  // namespace
}  // namespace mxa

extern "C" mxa_status mxa_bwd_noalloc(const mxa_bwd_params* p, cudaStream_t stream) {
  using namespace mxa;
  if (!p) return MXA_ERR_ARG;
  // mxa_bwd's own argument checks: given no workspace it validates every
  // argument and stops at MXA_ERR_WORKSPACE before any work, so an invalid
  // call gets exactly the status mxa_bwd would give it
  const mxa_status st = mxa_bwd(p, nullptr, 0, stream);
  if (st != MXA_ERR_WORKSPACE) return st;
  // the smallest workspace mxa_bwd accepts must fit; a call whose emitted dS
  // also fits takes the faster dQ path inside mxa_bwd
  const size_t need = mxa_bwd_workspace_min_bytes(p);
  if (need == 0 || need > MXA_BWD_NOALLOC_MAX_WORKSPACE) return MXA_ERR_WORKSPACE;
  // The array's address on the current device, looked up on every call (no
  // cache that a device reset could leave stale); the lookup allocates
  // nothing.  The first lookup on a device loads the module there.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_bwd_scratch) != cudaSuccess || scratch == nullptr) return MXA_ERR_CUDA;
  // mxa_bwd writes every byte it later reads (D and LSE rows, pad rows
  // included, the tile lists, the emitted dS of every visible tile pair) and
  // zeroes the fp16 dQ accumulator itself, so the contents a previous call
  // left behind never leak into this one.
  return mxa_bwd(p, scratch, MXA_BWD_NOALLOC_MAX_WORKSPACE, stream);
}
