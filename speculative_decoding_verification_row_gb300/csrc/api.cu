// C ABI of libspecverify.so: host-side validation, workspace carving and
// dispatch.  Every computation of the verification row runs in the kernels of
// chain.cu and argmax.cu; this file only checks arguments and launches.
#include <float.h>
#include <stddef.h>
#include <math.h>

#include "kernels.cuh"

namespace {

using namespace sv;

constexpr double kLog2e = 1.4426950408889634073599246810019;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int esize(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

// log2(e)/T as c_hi + c_lo with c_hi rounded down and c_lo > 0.
bool temperature_consts(float T, float* hi, float* lo, float* rn = nullptr) {
  if (!(T > 0.f) || !isfinite(T)) return false;
  const double c = kLog2e / (double)T;
  if (!(c < (double)FLT_MAX) || !(c > (double)FLT_MIN)) return false;
  float h = (float)c;
  if ((double)h > c) h = nextafterf(h, 0.f);
  float l = (float)(c - (double)h);
  if (!(l > 0.f)) l = FLT_MIN;
  *hi = h;
  *lo = l;
  if (rn) *rn = (float)c;
  return true;
}

// Units of one row: vectors per row, units per row and vectors per unit.
void row_units(int V, int dtype, bool vec, int* nvec, int* nsplit, int* vps) {
  *nvec = vec ? (int)((size_t)V * esize(dtype) / 16) : V;
  *nsplit = ceil_div(*nvec, kUnitVecs);
  *vps = ceil_div(*nvec, *nsplit);
}

int check_ws(void* ws, size_t bytes, int B, int rows, int V) {
  if (!ws || !aligned16(ws)) return SPEC_EWORKSPACE;
  if (bytes < WsLayout(B, rows, V).total) return SPEC_EWORKSPACE;
  return SPEC_OK;
}

__global__ void rollback_kernel(const int32_t* old_lens, const int32_t* n_acc, int k, int B,
                                int32_t* new_lens, int32_t* rewind_lens) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int32_t n = n_acc[b], old = old_lens[b];
  if (n < 0 || n > k) {  // a failed request or a corrupt count: length kept, rewind -1
    new_lens[b] = old;
    if (rewind_lens) rewind_lens[b] = -1;
    return;
  }
  new_lens[b] = old + n + 1;
  if (rewind_lens) rewind_lens[b] = k - n;
}

// Rollback with ragged draft lengths and paged block accounting: rewind =
// k_b - n, and the blocks past ceil(new_len / tokens_per_block) are free.
__global__ void rollback_paged_kernel(const int32_t* old_lens, const int32_t* n_acc,
                                      const int32_t* draft_lens, int k,
                                      const int32_t* blocks_held, int tpb, int B,
                                      int32_t* new_lens, int32_t* rewind_lens,
                                      int32_t* free_blocks) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int32_t kb = draft_lens ? draft_lens[b] : k, n = n_acc[b], old = old_lens[b];
  if (kb < 0 || kb > k || n < 0 || n > kb) {
    new_lens[b] = old;
    if (rewind_lens) rewind_lens[b] = -1;
    if (free_blocks) free_blocks[b] = 0;
    return;
  }
  const long long len = (long long)old + n + 1;
  new_lens[b] = (int32_t)len;
  if (rewind_lens) rewind_lens[b] = kb - n;
  if (free_blocks) {
    const long long spare = blocks_held ? blocks_held[b] - (len + tpb - 1) / tpb : 0;
    free_blocks[b] = spare > 0 ? (int32_t)spare : 0;
  }
}

}  // namespace

extern "C" {

size_t spec_workspace_size(int B, int rows_per_request, int V) {
  if (B < 1 || B > SPEC_MAX_BATCH || rows_per_request < 1 || V < 2) return 0;
  return WsLayout(B, rows_per_request, V).total;
}

size_t spec_workspace_size_filtered(int B, int k, int V, int top_k) {
  if (B < 1 || B > SPEC_MAX_BATCH || k < 1 || k > SPEC_MAX_DRAFT || V < 2 || top_k < 0)
    return 0;
  // top_k = 0 (top-p or min_p alone, or no filter) and top_k above
  // SPEC_MAX_TOPK take the per-row cuts of the wide path
  if (top_k == 0 || top_k > SPEC_MAX_TOPK) return WideLayout(B, k, V).total;
  return FilterLayout(B, k, V, top_k).total;
}

int spec_workspace_init(void* workspace, size_t workspace_bytes, spec_stream_t stream) {
  if (!workspace || workspace_bytes == 0) return SPEC_EINVAL;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) != cudaSuccess)
    return SPEC_ECUDA;
  return SPEC_OK;
}

}  // extern "C"

namespace sv {

// Checks the arguments of a chain verify (explicit uniforms, or with
// uniforms == nullptr each request's Philox (seed, offset)) and fills the
// launch arguments; launches nothing and writes nothing.
int chain_setup(ChainArgs& a, bool& vec, const void* target_logits, const void* draft_logits,
                int dtype, const int32_t* draft_tokens, const float* uniforms,
                const uint64_t* seeds, const uint64_t* offsets, const int32_t* draft_lens,
                float temperature, int B, int k, int V, int32_t* out_tokens,
                int32_t* out_num_accepted, float* out_probs, int32_t* seq_lens, void* workspace,
                size_t workspace_bytes, int top_k, float top_p, float min_p) {
  if (!target_logits || !draft_logits || !draft_tokens || (!uniforms && (!seeds || !offsets)) ||
      !out_tokens || !out_num_accepted)
    return SPEC_EINVAL;
  if ((dtype != SPEC_F32 && dtype != SPEC_BF16) || B < 1 || B > SPEC_MAX_BATCH || k < 1 ||
      k > SPEC_MAX_DRAFT || V < 2)
    return SPEC_EINVAL;
  a = ChainArgs{};
  if (!temperature_consts(temperature, &a.c_hi, &a.c_lo, &a.c_rn)) return SPEC_EINVAL;
  const int R = 2 * k + 1;
  if (top_k < 0 || !(top_p > 0.f) || !(top_p <= 1.f) || !(min_p >= 0.f) || !(min_p <= 1.f))
    return SPEC_EINVAL;
  // Kept lists for 1 <= top_k <= SPEC_MAX_TOPK; per-row cuts for kept sets
  // of any size (top-p or min_p without top-k, or a larger top-k).
  const bool wide = (top_k == 0 && (top_p < 1.f || min_p > 0.f)) || top_k > SPEC_MAX_TOPK;
  const int kcand = wide ? 0 : top_k;
  if (const int rc = check_ws(workspace, workspace_bytes, B, R, V)) return rc;
  vec = aligned16(target_logits) && aligned16(draft_logits) &&
        ((size_t)V * esize(dtype)) % 16 == 0;
  row_units(V, dtype, vec, &a.nvec, &a.nsplit, &a.vps);
  if (kcand > 0 && workspace_bytes < FilterLayout(B, k, V, kcand).total) return SPEC_EWORKSPACE;
  if (wide && workspace_bytes < WideLayout(B, k, V).total) return SPEC_EWORKSPACE;
  a.nchunks = num_chunks(V);
  a.cpc = kChunksPerCta;
  a.nsplit2 = num_items(V);
  if ((long)B * (R * (long)a.nsplit + a.nsplit2) > INT_MAX) return SPEC_EINVAL;  // grid sizes
  a.target = static_cast<const char*>(target_logits);
  a.draft = static_cast<const char*>(draft_logits);
  a.tokens = draft_tokens;
  a.uniforms = uniforms;
  a.seeds = reinterpret_cast<const unsigned long long*>(seeds);
  a.offsets = reinterpret_cast<const unsigned long long*>(offsets);
  a.draft_lens = draft_lens;
  a.B = B;
  a.k = k;
  a.V = V;
  a.rows = R;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.out_probs = out_probs;
  a.seq_lens = seq_lens;
  a.wait_cycles = kWaitCycles;
  a.ws = ws_views(workspace, WsLayout(B, R, V));
  a.top_k = wide ? top_k : kcand;
  a.top_p = top_p;
  a.min_p = min_p;
  a.wide = wide;
  if (wide) {
    const WideLayout wl(B, k, V);
    char* base = static_cast<char*>(workspace);
    a.ws.whist = reinterpret_cast<unsigned long long*>(base + wl.hist);
    a.ws.wcount = reinterpret_cast<unsigned*>(base + wl.count);
    a.ws.wrow = reinterpret_cast<WideRow*>(base + wl.rec);
    a.ws.wcand = reinterpret_cast<unsigned*>(base + wl.cand);
  } else if (kcand > 0) {
    const FilterLayout fl(B, k, V, kcand);
    a.ws.cand = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + fl.cand);
    a.ws.pq = reinterpret_cast<float*>(static_cast<char*>(workspace) + fl.pq);
    a.ws.codes = reinterpret_cast<unsigned short*>(static_cast<char*>(workspace) + fl.codes);
  }
  return SPEC_OK;
}

// Enqueues a chain verify set up by chain_setup.
int chain_launch(const ChainArgs& a, int dtype, bool vec, cudaStream_t st, bool skip_pass1) {
  if (a.wide && skip_pass1) return SPEC_EINVAL;  // the wide path waits for nothing
  const cudaError_t e = a.wide        ? launch_wide(a, dtype, vec, st)
                        : a.top_k > 0 ? launch_filtered(a, dtype, vec, st, skip_pass1)
                                      : launch_chain(a, dtype, vec, st, skip_pass1);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace sv

namespace {

int chain_impl(const void* target_logits, const void* draft_logits, int dtype,
               const int32_t* draft_tokens, const float* uniforms, const uint64_t* seeds,
               const uint64_t* offsets, const int32_t* draft_lens, float temperature, int B,
               int k, int V, int32_t* out_tokens, int32_t* out_num_accepted, float* out_probs,
               int32_t* seq_lens, void* workspace, size_t workspace_bytes, spec_stream_t stream,
               int top_k = 0, float top_p = 1.f, long long wait_cycles = kWaitCycles,
               bool skip_pass1 = false, float min_p = 0.f) {
  ChainArgs a;
  bool vec = false;
  if (const int rc = chain_setup(a, vec, target_logits, draft_logits, dtype, draft_tokens, uniforms,
                                 seeds, offsets, draft_lens, temperature, B, k, V, out_tokens,
                                 out_num_accepted, out_probs, seq_lens, workspace, workspace_bytes,
                                 top_k, top_p, min_p))
    return rc;
  a.wait_cycles = wait_cycles;
  return chain_launch(a, dtype, vec, (cudaStream_t)stream, skip_pass1);
}

__global__ void philox_uniforms_kernel(const unsigned long long* seeds,
                                       const unsigned long long* offsets, int B, int n,
                                       float* out) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)B * n) return;
  const int b = (int)(i / n);
  out[i] = philox_uniform(seeds[b], offsets[b], (int)(i - (long)b * n));
}

}  // namespace

extern "C" {

int spec_philox_uniforms(const uint64_t* seeds, const uint64_t* offsets, int B, int n,
                         float* out, spec_stream_t stream) {
  if (!seeds || !offsets || !out || B < 1 || B > SPEC_MAX_BATCH || n < 1 ||
      n > SPEC_MAX_DRAFT + 1)
    return SPEC_EINVAL;
  const long total = (long)B * n;
  philox_uniforms_kernel<<<(unsigned)((total + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const unsigned long long*>(seeds),
      reinterpret_cast<const unsigned long long*>(offsets), B, n, out);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_verify_chain(const void* target_logits, const void* draft_logits, int dtype,
                      const int32_t* draft_tokens, const float* uniforms, float temperature,
                      int B, int k, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                      float* out_probs, int32_t* seq_lens, void* workspace,
                      size_t workspace_bytes, spec_stream_t stream) {
  if (!uniforms) return SPEC_EINVAL;
  return chain_impl(target_logits, draft_logits, dtype, draft_tokens, uniforms, nullptr, nullptr,
                    nullptr, temperature, B, k, V, out_tokens, out_num_accepted, out_probs,
                    seq_lens, workspace, workspace_bytes, stream);
}

int spec_verify_chain_philox(const void* target_logits, const void* draft_logits, int dtype,
                             const int32_t* draft_tokens, const uint64_t* seeds,
                             const uint64_t* offsets, float temperature, int B, int k, int V,
                             int32_t* out_tokens, int32_t* out_num_accepted, float* out_probs,
                             int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream) {
  if (!seeds || !offsets) return SPEC_EINVAL;
  return chain_impl(target_logits, draft_logits, dtype, draft_tokens, nullptr, seeds, offsets,
                    nullptr, temperature, B, k, V, out_tokens, out_num_accepted, out_probs,
                    seq_lens, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

int greedy_impl(const void* target_logits, int dtype, const int32_t* draft_tokens,
                const int32_t* draft_lens, int B, int k, int V, int32_t* out_tokens,
                int32_t* out_num_accepted, int32_t* seq_lens, void* workspace,
                size_t workspace_bytes, spec_stream_t stream,
                long long wait_cycles = kWaitCycles, bool skip_pass1 = false) {
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted) return SPEC_EINVAL;
  if ((dtype != SPEC_F32 && dtype != SPEC_BF16) || B < 1 || B > SPEC_MAX_BATCH || k < 1 ||
      k > SPEC_MAX_DRAFT || V < 2)
    return SPEC_EINVAL;
  const int R = k + 1;
  if (const int rc = check_ws(workspace, workspace_bytes, B, R, V)) return rc;
  ArgmaxArgs a{};
  const bool vec = aligned16(target_logits) && ((size_t)V * esize(dtype)) % 16 == 0;
  row_units(V, dtype, vec, &a.nvec, &a.nsplit, &a.vps);
  if ((long)B * R * a.nsplit > INT_MAX) return SPEC_EINVAL;
  a.target = static_cast<const char*>(target_logits);
  a.B = B;
  a.R = R;
  a.V = V;
  a.tree = 0;
  a.draft_tokens = draft_tokens;
  a.draft_lens = draft_lens;
  a.k = k;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.seq_lens = seq_lens;
  a.wait_cycles = wait_cycles;
  a.ws = ws_views(workspace, WsLayout(B, R, V));
  return launch_argmax(a, dtype, vec, (cudaStream_t)stream, skip_pass1) == cudaSuccess
             ? SPEC_OK
             : SPEC_ECUDA;
}

}  // namespace

extern "C" {

int spec_verify_greedy(const void* target_logits, int dtype, const int32_t* draft_tokens, int B,
                       int k, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                       int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                       spec_stream_t stream) {
  return greedy_impl(target_logits, dtype, draft_tokens, nullptr, B, k, V, out_tokens,
                     out_num_accepted, seq_lens, workspace, workspace_bytes, stream);
}

int spec_verify_greedy_ex(const spec_greedy_params* p, void* workspace, size_t workspace_bytes,
                          spec_stream_t stream) {
  if (!p || p->size < sizeof(spec_greedy_params)) return SPEC_EINVAL;
  return greedy_impl(p->target_logits, p->dtype, p->draft_tokens, p->draft_lens, p->B, p->k,
                     p->V, p->out_tokens, p->out_num_accepted, p->seq_lens, workspace,
                     workspace_bytes, stream);
}

int spec_verify_chain_ex(const spec_chain_params* p, void* workspace, size_t workspace_bytes,
                         spec_stream_t stream) {
  // Earlier versions of the struct end at seq_lens (no filtering fields) or
  // at top_p (no min_p).
  const size_t v1 = offsetof(spec_chain_params, seq_lens) + sizeof(p->seq_lens);
  if (!p || p->size < v1) return SPEC_EINVAL;
  const bool has_filter = p->size >= offsetof(spec_chain_params, top_p) + sizeof(p->top_p);
  const bool has_min_p = p->size >= offsetof(spec_chain_params, min_p) + sizeof(p->min_p);
  return chain_impl(p->target_logits, p->draft_logits, p->dtype, p->draft_tokens, p->uniforms,
                    p->seeds, p->offsets, p->draft_lens, p->temperature, p->B, p->k, p->V,
                    p->out_tokens, p->out_num_accepted, p->out_probs, p->seq_lens, workspace,
                    workspace_bytes, stream, has_filter ? p->top_k : 0,
                    has_filter ? p->top_p : 1.f, kWaitCycles, false,
                    has_min_p ? p->min_p : 0.f);
}

int spec_test_timeout_chain(const spec_chain_params* p, long long wait_cycles, void* workspace,
                            size_t workspace_bytes, spec_stream_t stream) {
  const size_t v1 = offsetof(spec_chain_params, seq_lens) + sizeof(p->seq_lens);
  if (!p || p->size < v1 || wait_cycles < 1) return SPEC_EINVAL;
  const bool has_filter = p->size >= offsetof(spec_chain_params, top_p) + sizeof(p->top_p);
  const bool has_min_p = p->size >= offsetof(spec_chain_params, min_p) + sizeof(p->min_p);
  return chain_impl(p->target_logits, p->draft_logits, p->dtype, p->draft_tokens, p->uniforms,
                    p->seeds, p->offsets, p->draft_lens, p->temperature, p->B, p->k, p->V,
                    p->out_tokens, p->out_num_accepted, p->out_probs, p->seq_lens, workspace,
                    workspace_bytes, stream, has_filter ? p->top_k : 0,
                    has_filter ? p->top_p : 1.f, wait_cycles, true, has_min_p ? p->min_p : 0.f);
}

int spec_test_timeout_greedy(const spec_greedy_params* p, long long wait_cycles, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream) {
  if (!p || p->size < sizeof(spec_greedy_params) || wait_cycles < 1) return SPEC_EINVAL;
  return greedy_impl(p->target_logits, p->dtype, p->draft_tokens, p->draft_lens, p->B, p->k,
                     p->V, p->out_tokens, p->out_num_accepted, p->seq_lens, workspace,
                     workspace_bytes, stream, wait_cycles, true);
}

int spec_rollback_paged(const int32_t* old_lens, const int32_t* num_accepted,
                        const int32_t* draft_lens, int k, const int32_t* blocks_held,
                        int tokens_per_block, int B, int32_t* new_lens, int32_t* rewind_lens,
                        int32_t* free_blocks, spec_stream_t stream) {
  if (!old_lens || !num_accepted || !new_lens || B < 1 || B > SPEC_MAX_BATCH || k < 0 ||
      tokens_per_block < 1)
    return SPEC_EINVAL;
  rollback_paged_kernel<<<ceil_div(B, 256), 256, 0, (cudaStream_t)stream>>>(
      old_lens, num_accepted, draft_lens, k, blocks_held, tokens_per_block, B, new_lens,
      rewind_lens, free_blocks);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_verify_tree(const void* target_logits, int dtype, const int32_t* tree_tokens,
                     const int32_t* paths, int B, int N, int P, int L, int V,
                     int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_best_path,
                     int32_t* out_accepted_nodes, int32_t* seq_lens, void* workspace,
                     size_t workspace_bytes, spec_stream_t stream) {
  if (!target_logits || !tree_tokens || !paths || !out_tokens || !out_num_accepted)
    return SPEC_EINVAL;
  if ((dtype != SPEC_F32 && dtype != SPEC_BF16) || B < 1 || B > SPEC_MAX_BATCH || N < 1 ||
      N > SPEC_MAX_TREE_NODES ||
      P < 1 || L < 2 || L > SPEC_MAX_PATH_LEN || V < 2 || (long)P * L > INT_MAX)
    return SPEC_EINVAL;
  if (const int rc = check_ws(workspace, workspace_bytes, B, N, V)) return rc;
  ArgmaxArgs a{};
  const bool vec = aligned16(target_logits) && ((size_t)V * esize(dtype)) % 16 == 0;
  row_units(V, dtype, vec, &a.nvec, &a.nsplit, &a.vps);
  if ((long)B * N * a.nsplit > INT_MAX) return SPEC_EINVAL;
  a.target = static_cast<const char*>(target_logits);
  a.B = B;
  a.R = N;
  a.V = V;
  a.tree = 1;
  a.tree_tokens = tree_tokens;
  a.paths = paths;
  a.P = P;
  a.L = L;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.out_best = out_best_path;
  a.out_nodes = out_accepted_nodes;
  a.seq_lens = seq_lens;
  a.wait_cycles = kWaitCycles;
  a.ws = ws_views(workspace, WsLayout(B, N, V));
  return launch_argmax(a, dtype, vec, (cudaStream_t)stream) == cudaSuccess ? SPEC_OK
                                                                           : SPEC_ECUDA;
}

int spec_verify_tree_sampled(const void* target_logits, int dtype, const int32_t* tree_tokens,
                             const int32_t* paths, const float* uniforms, float temperature, int B,
                             int N, int P, int L, int V, int32_t* out_tokens,
                             int32_t* out_num_accepted, int32_t* out_best_path,
                             int32_t* out_accepted_nodes, int32_t* seq_lens, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream) {
  if (!target_logits || !tree_tokens || !paths || !uniforms || !out_tokens || !out_num_accepted)
    return SPEC_EINVAL;
  if ((dtype != SPEC_F32 && dtype != SPEC_BF16) || B < 1 || B > SPEC_MAX_BATCH || N < 1 ||
      N > SPEC_MAX_TREE_NODES || P < 1 || L < 2 || L > SPEC_MAX_PATH_LEN || V < 2 ||
      (long)P * L > kTreeStage)
    return SPEC_EINVAL;
  ChainArgs a{};
  if (!temperature_consts(temperature, &a.c_hi, &a.c_lo, &a.c_rn)) return SPEC_EINVAL;
  if (const int rc = check_ws(workspace, workspace_bytes, B, N, V)) return rc;
  const bool vec = aligned16(target_logits) && ((size_t)V * esize(dtype)) % 16 == 0;
  row_units(V, dtype, vec, &a.nvec, &a.nsplit, &a.vps);
  a.nchunks = num_chunks(V);
  a.cpc = kChunksPerCta;
  a.nsplit2 = num_items(V);
  if ((long)B * ((long)N * a.nsplit + a.nsplit2) > INT_MAX) return SPEC_EINVAL;  // grid sizes
  a.target = static_cast<const char*>(target_logits);
  a.uniforms = uniforms;
  a.B = B;
  a.k = N - 1;  // pass 1 reads target rows 0..N-1
  a.V = V;
  a.rows = N;
  a.tree_tokens = tree_tokens;
  a.paths = paths;
  a.P = P;
  a.L = L;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.out_best = out_best_path;
  a.out_nodes = out_accepted_nodes;
  a.seq_lens = seq_lens;
  a.wait_cycles = kWaitCycles;
  a.ws = ws_views(workspace, WsLayout(B, N, V));
  return launch_tree_sampled(a, dtype, vec, (cudaStream_t)stream) == cudaSuccess ? SPEC_OK
                                                                                 : SPEC_ECUDA;
}

int spec_rollback_lengths(const int32_t* old_lens, const int32_t* num_accepted, int k, int B,
                          int32_t* new_lens, int32_t* rewind_lens, spec_stream_t stream) {
  if (!old_lens || !num_accepted || !new_lens || B < 1 || k < 0) return SPEC_EINVAL;
  rollback_kernel<<<ceil_div(B, 256), 256, 0, (cudaStream_t)stream>>>(old_lens, num_accepted, k,
                                                                       B, new_lens, rewind_lens);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_last_error(void* workspace, size_t workspace_bytes, spec_stream_t stream,
                    int* status_out) {
  if (!workspace || !status_out || workspace_bytes < sizeof(int)) return SPEC_EINVAL;
  const cudaStream_t st = (cudaStream_t)stream;
  int h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess)
    return SPEC_ECUDA;
  *status_out = h;
  return SPEC_OK;
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument";
    case SPEC_EBADINDEX: return "token or node id out of range";
    case SPEC_ECUDA: return "CUDA error";
    case SPEC_EWORKSPACE: return "workspace missing or too small";
    case SPEC_ETIMEOUT: return "device wait timed out";
    case SPEC_ELIMIT: return "a filtered row's cut search failed an internal check";
    default: return "unknown status";
  }
}

}  // extern "C"
