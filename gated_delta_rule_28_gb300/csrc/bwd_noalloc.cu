// Backward entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: runtimes that plan every device
// buffer when they start and forbid allocation afterwards, and plugin hosts
// that hand a library its input and output buffers but no allocator. For
// them, gdn_chunk_bwd_noalloc runs the same backward as gdn_chunk_bwd with
// its scratch memory in a fixed array inside this library instead of a
// caller-provided workspace.
//
// The array below is a file-scope device variable: every GPU that loads the
// library holds GDN_NOALLOC_SCRATCH_BYTES of device memory for it until the
// process exits. In host code its name is only a host-side stand-in, so every
// call looks up the array's device address on the current device with
// cudaGetSymbolAddress and passes that address to the kernels. The lookup is
// cheap and never cached, so an address can never outlive a device reset.
#include <cuda_runtime.h>

#include <cstdio>

#include "../../include/gdn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)GDN_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" gdn_status gdn_chunk_bwd_noalloc(const gdn_problem *p, const void *q, const void *k,
                                            const void *v, const float *g_cumsum, const void *beta,
                                            const float *A, const void *dO, const float *h0,
                                            const float *dht, void *dq, void *dk, void *dv,
                                            float *dg, void *dbeta, float *dh0, void *stream) {
  // the scratch this problem needs: the layout gdn_chunk_bwd uses
  size_t need = 0;
  gdn_status st = gdn_chunk_bwd_workspace(p, &need);
  if (st != GDN_OK) return st;
  char msg[256];
  if (need > kScratchBytes) {
    snprintf(msg, sizeof(msg),
             "gdn_chunk_bwd_noalloc: this problem needs %zu bytes of scratch; the built-in array "
             "holds %zu bytes (use gdn_chunk_bwd with a caller-provided workspace)",
             need, kScratchBytes);
    return gdn::set_error(GDN_ERR_WORKSPACE, msg);
  }
  // device address of the array on the current device, looked up on every call
  void *scratch = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
  if (e != cudaSuccess || !scratch) {
    snprintf(msg, sizeof(msg), "gdn_chunk_bwd_noalloc: scratch address lookup failed: %s",
             cudaGetErrorString(e));
    return gdn::set_error(GDN_ERR_CUDA, msg);
  }
  return gdn_chunk_bwd(p, q, k, v, g_cumsum, beta, A, dO, h0, dht, dq, dk, dv, dg, dbeta, dh0,
                       scratch, kScratchBytes, stream);
}
