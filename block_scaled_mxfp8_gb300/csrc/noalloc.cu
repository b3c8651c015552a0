// noalloc.cu -- mxa_bwd_noalloc: the backward pass with its scratch space in a
// device array that the library itself owns, for callers that cannot allocate
// device memory (see include/mxa.h).  This file adds one entry point and
// changes no existing code path: it resolves the array's device address and
// hands it to mxa_bwd as the workspace.
#include <mutex>

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

std::mutex g_scratch_mu;
void* g_scratch_addr[64];  // per device, resolved on the first call made with that device current

}  // namespace
}  // namespace mxa

extern "C" mxa_status mxa_bwd_noalloc(const mxa_bwd_params* p, cudaStream_t stream) {
  using namespace mxa;
  if (!p) return MXA_ERR_ARG;
  // the smallest workspace mxa_bwd accepts must fit; a call whose emitted dS
  // also fits takes the faster dQ path inside mxa_bwd
  const size_t need = mxa_bwd_workspace_min_bytes(p);
  if (need == 0) return MXA_ERR_ARG;
  if (need > MXA_BWD_NOALLOC_MAX_WORKSPACE) return MXA_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MXA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_bwd_scratch) != cudaSuccess || addr == nullptr) return MXA_ERR_CUDA;
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  // mxa_bwd writes every byte it later reads (D and LSE rows, pad rows
  // included, the emitted dS of every visible tile pair) and zeroes the fp16
  // dQ accumulator itself, so the contents a previous call left behind never
  // leak into this one.
  return mxa_bwd(p, scratch, MXA_BWD_NOALLOC_MAX_WORKSPACE, stream);
}
