// spec_verify_chain_noalloc: chain verify for callers that cannot allocate
// device memory (for example code running under an allocator that forbids
// allocations during a step, or host code that owns no CUDA allocator).  The
// scratch it needs lives in a file-scope device array of fixed size, present
// on every GPU that loads this library until the process exits.
#include "kernels.cuh"

namespace {

using namespace sv;

// Zero-initialised at module load; shared by every call on the device.
__device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

// The array's device address on the current device and context.  Host code
// only sees a host-side stand-in for the symbol, so the address is looked up
// on every call (a cheap runtime query): a cached address could outlive a
// device reset or belong to another context.
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ECUDA;
  *out = p;
  return SPEC_OK;
}

// Device memory of the current device (or managed memory).
bool on_current_device(const void* ptr, int dev) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();  // clear this (non-sticky) error so later launch checks do not see it
    return false;
  }
  if (attr.type == cudaMemoryTypeManaged) return true;
  return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}

}  // namespace

extern "C" int spec_verify_chain_noalloc(const void* target_logits, const void* draft_logits,
                                         int dtype, const int32_t* draft_tokens,
                                         const float* uniforms, float temperature, int B, int k,
                                         int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                         float* out_probs, int32_t* seq_lens,
                                         spec_stream_t stream) {
  if (B < 1 || B > SPEC_MAX_BATCH || k < 1 || k > SPEC_MAX_DRAFT || V < 2 || !uniforms)
    return SPEC_EINVAL;
  const WsLayout layout(B, 2 * k + 1, V);
  if (layout.total > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_EWORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  void* scratch = nullptr;
  if (const int rc = scratch_address(&scratch)) return rc;
  // Every argument is checked before the shared array is written, so a call
  // that is refused cannot disturb another call still using it.
  ChainArgs a;
  bool vec = false;
  if (const int rc = chain_setup(a, vec, target_logits, draft_logits, dtype, draft_tokens,
                                 uniforms, nullptr, nullptr, nullptr, temperature, B, k, V,
                                 out_tokens, out_num_accepted, out_probs, seq_lens, scratch,
                                 SPEC_NOALLOC_SCRATCH_BYTES, 0, 1.f, 0.f))
    return rc;
  // The kernels run on the current device, whose array this is: the caller's
  // arrays must live there too.
  const void* arrays[] = {target_logits, draft_logits, draft_tokens, uniforms, out_tokens,
                          out_num_accepted, out_probs, seq_lens};
  for (const void* p : arrays)
    if (p && !on_current_device(p, dev)) return SPEC_EINVAL;
  // The status word, this call's sync lines and its slice-statistics words
  // must start at zero; the rest is written before it is read within the
  // call.
  if (cudaMemsetAsync(scratch, 0, layout.sync + sizeof(ReqSync) * (size_t)B,
                      (cudaStream_t)stream) != cudaSuccess ||
      cudaMemsetAsync(static_cast<char*>(scratch) + layout.stats, 0,
                      stats_bytes(B, 2 * k + 1, V), (cudaStream_t)stream) != cudaSuccess)
    return SPEC_ECUDA;
  return chain_launch(a, dtype, vec, (cudaStream_t)stream, false);
}
