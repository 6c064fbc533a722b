// vqkv_decode_attn_static: the decode entry point for callers that cannot
// allocate device memory.  Same kernels and same results as
// vqkv_decode_attn, but the split-KV scratch (error word, per-(sequence, KV
// head) tickets, split partials) lives in a fixed array compiled into this
// library instead of a caller-provided workspace.
#include "internal.h"
#include "vqkv.h"

namespace vqkv {
namespace {

// Scratch of the allocation-free decode.  Every GPU that loads the library
// holds it until the process exits.  Zero-initialised at load; each call
// clears the error word and the tickets before launching.
static __device__ __align__(256) unsigned char g_decode_scratch[VQKV_STATIC_SCRATCH_BYTES];

// Device address of the scratch array in the current device's context.  It
// is looked up on every call (with the device current): the lookup
// allocates nothing, and a fresh lookup stays right after the context has
// been torn down and rebuilt (cudaDeviceReset), where a cached address
// would point into the old context.  The first lookup in a context may load
// the library's device code into it.
vqkv_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return VQKV_ERR_CUDA;
  *out = p;
  return VQKV_OK;
}

}  // namespace
}  // namespace vqkv

extern "C" vqkv_status vqkv_decode_attn_static(const vqkv_decode_args* args, void* stream) {
  using namespace vqkv;
  // every argument check first: a failed check enqueues nothing
  vqkv_status st = decode_validate(args);
  if (st != VQKV_OK || args->B == 0) return st;
  const size_t need = vqkv_decode_workspace_bytes(args);
  if (need == 0) return VQKV_ERR_NO_DEVICE;
  if (need > (size_t)VQKV_STATIC_SCRATCH_BYTES) return VQKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != VQKV_OK) return st;
  // the error word and the tickets must start at zero
  if (cudaMemsetAsync(scratch, 0, decode_ticket_region_bytes(args->B, args->Hkv),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VQKV_ERR_CUDA;
  vqkv_decode_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = VQKV_STATIC_SCRATCH_BYTES;
  return vqkv_decode_attn(&a, stream);
}

extern "C" vqkv_status vqkv_decode_static_error(uint32_t* host_flags, void* stream) {
  using namespace vqkv;
  if (host_flags == nullptr) return VQKV_ERR_INVALID_ARG;
  void* scratch = nullptr;
  vqkv_status st = scratch_address(&scratch);
  if (st != VQKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return VQKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return VQKV_ERR_CUDA;
  return VQKV_OK;
}
