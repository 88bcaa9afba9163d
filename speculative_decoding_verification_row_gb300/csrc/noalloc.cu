// spec_verify_chain_noalloc: chain verify for callers that cannot allocate
// device memory (for example code running under an allocator that forbids
// allocations during a step, or host code that owns no CUDA allocator).  The
// scratch it needs lives in a file-scope device array of fixed size, present
// on every GPU that loads this library until the process exits.
#include <mutex>

#include "kernels.cuh"

namespace {

using namespace sv;

constexpr int kMaxDevices = 64;

// Zero-initialised at module load; shared by every call on the device.
__device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code only sees a host-side stand-in for the symbol).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_EINVAL;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_chain_noalloc(const void* target_logits, const void* draft_logits,
                                         int dtype, const int32_t* draft_tokens,
                                         const float* uniforms, float temperature, int B, int k,
                                         int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                         float* out_probs, int32_t* seq_lens,
                                         spec_stream_t stream) {
  if (B < 1 || B > SPEC_MAX_BATCH || k < 1 || k > SPEC_MAX_DRAFT || V < 2) return SPEC_EINVAL;
  const WsLayout layout(B, 2 * k + 1, V);
  if (layout.total > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_EWORKSPACE;
  void* scratch = nullptr;
  if (const int rc = scratch_address(&scratch)) return rc;
  // The status word, this call's sync lines and its slice-statistics words
  // must start at zero; the rest is written before it is read within the
  // call.
  if (cudaMemsetAsync(scratch, 0, layout.sync + sizeof(ReqSync) * (size_t)B,
                      (cudaStream_t)stream) != cudaSuccess ||
      cudaMemsetAsync(static_cast<char*>(scratch) + layout.stats, 0,
                      stats_bytes(B, 2 * k + 1, V), (cudaStream_t)stream) != cudaSuccess)
    return SPEC_ECUDA;
  return spec_verify_chain(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                           temperature, B, k, V, out_tokens, out_num_accepted, out_probs,
                           seq_lens, scratch, SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
