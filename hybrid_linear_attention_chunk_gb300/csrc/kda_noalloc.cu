// kda_chunk_fwd_noalloc: kda_chunk_fwd for callers that cannot allocate
// device memory (see include/kda.h).  The workspace of the long-sequence
// plan comes from a fixed array compiled into the library instead of from
// cudaMallocAsync or from the caller.
#include "kda_internal.cuh"

namespace kda {
namespace {

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[KDA_STATIC_WORKSPACE_BYTES];

// Device address of g_static_ws in the current device's context.  In host
// code the name g_static_ws is only a host-side stand-in, so the address is
// looked up with that device current.  It is looked up on every call and not
// cached: a context that is destroyed and created again (cudaDeviceReset, a
// primary context released and retained) loads the module again, and the
// array may then sit at another address.  The lookup allocates nothing.
kda_status static_ws_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return KDA_ERR_CUDA;
  *out = p;
  return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_chunk_fwd_noalloc(const kda_chunk_desc *desc, const void *q, const void *k,
                                            const void *v, const void *log_alpha, const void *beta,
                                            const float *initial_state, const int32_t *cu_seqlens, void *out,
                                            float *final_state, kda_stream_t stream) {
  if (!desc) return KDA_ERR_NULL;
  if (desc->validate) return KDA_ERR_UNSUPPORTED;  // its range check would need an allocation
  size_t need = 0;
  kda_status st = kda_chunk_fwd_workspace_size(desc, &need);
  if (st != KDA_OK) return st;
  if (need > KDA_STATIC_WORKSPACE_BYTES) return KDA_ERR_SCRATCH_LIMIT;
  void *ws = nullptr;
  if (need > 0) {
    st = kda::static_ws_address(&ws);
    if (st != KDA_OK) return st;
  }
  // The segment passes write every workspace byte they later read, so the
  // previous call's contents need no clearing.
  return kda_chunk_fwd_ex(desc, q, k, v, log_alpha, beta, initial_state, cu_seqlens, out, final_state, ws,
                          need > 0 ? (size_t)KDA_STATIC_WORKSPACE_BYTES : 0, stream);
}
